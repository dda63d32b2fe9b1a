// control.cu -- integer kernels of the lookahead step: row assembly with the
// pool lookup, greedy (or sampling) verification + n-gram harvest + window
// shift, KV commit, and the GPU n-gram pool (hash table) with
// warp-cooperative lookup/insert.
//
// Method: Fu et al. 2024, "Break the Sequential Dependency of LLM Inference
// Using Lookahead Decoding" (summary page, "Summary"): a lookahead branch over
// a 2D window of W columns x (N-1) levels produces n-grams that are cached in
// a pool; a verification branch checks pool candidates in the same forward
// pass so that the output stays exactly the greedy output.
#include <climits>

#include "../../include/lookahead.h"
#include "common.cuh"

namespace la {

// ------------------------------------------------------------------ pool ---

__device__ __forceinline__ int pool_hash(const PoolView& p, int key)
{
    return (int)(((unsigned)key * 2654435761u) >> (32 - p.log2cap));
}

// Warp-cooperative probe (linear probing, 32 slots per round).  Returns the
// slot holding key (*found = true) or the first empty slot where it would go
// (*found = false); -1 if the table is full.  Keys are never deleted, so the
// first slot that holds either the key or -1 ends the probe.
__device__ int pool_probe(const PoolView& p, int key, bool* found)
{
    const int lane = threadIdx.x & 31;
    const int h = pool_hash(p, key);
    for (int base = 0; base < p.cap; base += 32) {
        int s = (h + base + lane) & (p.cap - 1);
        int k = p.keys[s];
        unsigned hit = __ballot_sync(0xffffffffu, k == key || k == -1);
        if (hit) {
            int src = __ffs(hit) - 1;
            int ks = __shfl_sync(0xffffffffu, k, src);
            *found = (ks == key);
            return (h + base + src) & (p.cap - 1);
        }
    }
    *found = false;
    return -1;
}

// Find or claim the slot of key with atomicCAS (concurrent warps).
__device__ int pool_claim(const PoolView& p, int key)
{
    const int lane = threadIdx.x & 31;
    int start = pool_hash(p, key);
    for (int probed = 0; probed < p.cap;) {
        int s = (start + lane) & (p.cap - 1);
        int k = p.keys[s];
        unsigned hit = __ballot_sync(0xffffffffu, k == key || k == -1);
        if (!hit) {
            start += 32;
            probed += 32;
            continue;
        }
        int src = __ffs(hit) - 1;
        int slot = (start + src) & (p.cap - 1);
        int old = 0;
        if (lane == src) old = (k == key) ? key : atomicCAS(&p.keys[slot], -1, key);
        old = __shfl_sync(0xffffffffu, old, src);
        if (old == key || old == -1) return slot;
        // another key took the slot first: continue from that slot
        start = slot;
        probed += src;
    }
    return -1;
}

// Insert the (n1)-gram val (held by every lane) into slot s: no-op if held,
// else append, evicting the oldest entry when G are held.  One warp per slot.
__device__ void pool_insert_slot(const PoolView& p, int s, const int* val)
{
    const int lane = threadIdx.x & 31;
    const int n1 = p.n1, G = p.G;
    int* ent = p.ent + (size_t)s * G * n1;
    int cnt = p.cnt[s];
    bool dup = false;
    for (int g0 = 0; g0 < cnt; g0 += 32) {
        int g = g0 + lane;
        bool eq = g < cnt;
        for (int i = 0; i < n1 && eq; i++) eq = (ent[g * n1 + i] == val[i]);
        if (__any_sync(0xffffffffu, eq)) dup = true;
    }
    if (dup) return;
    if (cnt == G) {
        // shift entries 1..G-1 down by one (read all, then write)
        int tmp[kMaxN * 4];
        int nread = 0;
        for (int idx = lane; idx < (G - 1) * n1; idx += 32) tmp[nread++] = ent[idx + n1];
        __syncwarp();
        nread = 0;
        for (int idx = lane; idx < (G - 1) * n1; idx += 32) ent[idx] = tmp[nread++];
        __syncwarp();
        cnt = G - 1;
    }
    if (lane < n1) ent[cnt * n1 + lane] = val[lane];
    __syncwarp();
    if (lane == 0) p.cnt[s] = cnt + 1;
    __syncwarp();
}

__global__ void k_pool_reset(PoolView p)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.cap; i += gridDim.x * blockDim.x) {
        p.keys[i] = -1;
        p.cnt[i] = 0;
        p.first[i] = INT_MAX;
    }
}

// bulk insert, phase 1: every insert finds/claims its key's slot; the lowest
// insert index of each slot becomes that key's leader.  Keys below 0 (-1 is
// the empty-slot marker) are refused: status LA_ERR_ARG, the insert skipped.
__global__ void k_pool_claim(PoolView p, const int* keys, int n)
{
    int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= n) return;
    const int key = keys[w];
    if (key < 0) {
        if ((threadIdx.x & 31) == 0) {
            p.slot_of[w] = -1;
            atomicCAS(p.status, 0, LA_ERR_ARG);
        }
        return;
    }
    int s = pool_claim(p, key);
    if ((threadIdx.x & 31) == 0) {
        p.slot_of[w] = s;
        if (s < 0) atomicCAS(p.status, 0, LA_ERR_CAPACITY);
        else atomicMin(&p.first[s], w);
    }
}

// bulk insert, phase 2: each key's leader warp applies that key's inserts in
// index order, so the result equals inserting all n in index order.
__global__ void k_pool_apply(PoolView p, const int* keys, const int* grams, int stride, int n)
{
    int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= n) return;
    int s = p.slot_of[w];
    if (s < 0 || p.first[s] != w) return;
    const int key = keys[w];
    int val[kMaxN];
    for (int j0 = w; j0 < n; j0 += 32) {
        int j = j0 + lane;
        unsigned m = __ballot_sync(0xffffffffu, j < n && keys[j] == key);
        while (m) {
            int b = __ffs(m) - 1;
            m &= m - 1;
            const int* g = grams + (size_t)(j0 + b) * stride;
            for (int i = 0; i < p.n1; i++) val[i] = g[i];
            pool_insert_slot(p, s, val);
        }
    }
    if (lane == 0) p.first[s] = INT_MAX;
}

__global__ void k_pool_lookup(PoolView p, const int* keys, int n, int* out, int* counts)
{
    int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= n) return;
    bool found = false;
    // a negative key is never held (-1 marks empty slots): absent
    int s = keys[w] >= 0 ? pool_probe(p, keys[w], &found) : -1;
    int cnt = (found && s >= 0) ? p.cnt[s] : 0;
    const int tot = p.G * p.n1;
    for (int i = lane; i < tot; i += 32)
        out[(size_t)w * tot + i] = (i < cnt * p.n1) ? p.ent[(size_t)s * tot + i] : -1;
    if (lane == 0) counts[w] = cnt;
}

void launch_pool_reset(cudaStream_t s, PoolView pool)
{
    k_pool_reset<<<ceil_div(pool.cap, 256), 256, 0, s>>>(pool);
}

void launch_pool_insert(cudaStream_t s, PoolView pool, const int* keys, const int* grams, int gram_stride, int n)
{
    if (n <= 0 || pool.G == 0) return;
    int blocks = ceil_div(n * 32, 256);
    k_pool_claim<<<blocks, 256, 0, s>>>(pool, keys, n);
    k_pool_apply<<<blocks, 256, 0, s>>>(pool, keys, grams, gram_stride, n);
}

void launch_pool_lookup(cudaStream_t s, PoolView pool, const int* keys, int n, int* out, int* counts)
{
    if (n <= 0) return;
    k_pool_lookup<<<ceil_div(n * 32, 256), 256, 0, s>>>(pool, keys, n, out, counts);
}

// ------------------------------------------------------------- step rows ---

// Rows of the step (row 0 = c; lookahead row (l,j) = 1 + l*W + j holds
// win[l][j]; verification row (g,i) = 1 + W(N-1) + g(N-1) + i holds the g-th
// candidate's i-th token), positions P + rel_pos[r].  Candidates are the pool
// entries of c, oldest first; missing candidates' rows are padding (token 0).
// Batched (gridDim.x = B > 1): block b builds sequence b's T rows only.
__global__ void k_build_rows(DState* st, const int* win, PoolView pool, int W, int N, int G, int T,
                             const int* rel_pos, int* tok, int* pos, size_t sb)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int s_slot, s_cnt;
    const int b = blockIdx.x;
    st = seq_ptr(st, sb, b);
    win = seq_ptr(win, sb, b);
    pool = seq_pool(pool, sb, b);
    tok += (size_t)b * T;
    pos += (size_t)b * T;
    const int nrows = gridDim.x > 1 ? T : kRows;
    const int c = st->c, P = st->P;
    if (threadIdx.x < 32) {
        bool found = false;
        int s = (G > 0) ? pool_probe(pool, c, &found) : -1;
        if (threadIdx.x == 0) {
            s_slot = (found && s >= 0) ? s : -1;
            s_cnt = (found && s >= 0) ? pool.cnt[s] : 0;
        }
    }
    __syncthreads();
    const int n1 = N - 1, slot = s_slot, cnt = s_cnt;
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
        int t = 0;
        if (r == 0) {
            t = c;
        } else if (r < 1 + W * n1) {
            t = win[r - 1];
        } else if (r < T) {
            int q = r - 1 - W * n1, g = q / n1, i = q - g * n1;
            t = (g < cnt) ? pool.ent[((size_t)slot * G + g) * n1 + i] : 0;
        }
        tok[r] = t;
        pos[r] = P + rel_pos[r];
    }
    if (threadIdx.x == 0) {
        st->ncand = cnt;
        st->T = T;
    }
}

void launch_build_rows(cudaStream_t s, DState* st, const int* win, PoolView pool, int W, int N, int G, int T,
                       const int* rel_pos, int* tok, int* pos, int B, size_t sb)
{
    launch_pdl(k_build_rows, dim3(B), dim3(128), 0, s, st, win, pool, W, N, G, T, rel_pos, tok, pos, sb);
}

__global__ void k_prefill_rows(const DState* st, const int* prompt, int P0, int n, int* tok, int* pos)
{
    for (int r = threadIdx.x; r < kRows; r += blockDim.x) {
        tok[r] = (r < n) ? prompt[P0 + r] : 0;
        pos[r] = P0 + ((r < n) ? r : 0);
    }
}

void launch_prefill_rows(cudaStream_t s, const DState* st, const int* prompt, int P0, int n, int* tok, int* pos)
{
    k_prefill_rows<<<1, 128, 0, s>>>(st, prompt, P0, n, tok, pos);
}


// ------------------------------------------------- sampling verification ---
//
// The summary page says the method supports sampling and keeps the output
// distribution; it gives no algorithm.  The rule used here: p = softmax(z /
// tau) of a row.  At each level, the distinct values of the still-matching
// candidates are tried in candidate order, value v accepted with probability
// p(v) / (1 - mass of the values already rejected at this level); if none is
// accepted the token is drawn from p without the rejected values.  The
// acceptance probabilities telescope, so every emitted token is distributed
// exactly as its row's softmax.  After the last level a bonus token is drawn
// from the last accepted row.  One uniform per candidate try and one per
// drawn token, in that order, from a splitmix64 stream in the decode state.

// splitmix64 (S. Vigna's published generator): add the golden gamma, then
// two xor-shift-multiply rounds and a final xor-shift.
__device__ __forceinline__ unsigned long long smix64(unsigned long long* x)
{
    unsigned long long z = (*x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}


// exp(x) for x <= 0 in fp32 for the sampling probabilities: range reduction
// after Cody and Waite, k = nearest integer to x log2(e), t = x - k ln 2 with
// ln 2 split into a float and its float remainder (two fused multiply-adds),
// e^x = 2^k e^t; e^t by its degree-7 Taylor series (Horner, fused
// multiply-adds), times 2^k; 0 below 2^-125.  Each step is one correctly
// rounded fp32 operation (no contraction left to the compiler), so the
// result does not depend on the device or the compiler.
__device__ __forceinline__ float exp_neg(float x)
{
    const float k = rintf(__fmul_rn(x, 0x1.715476p+0f));
    if (k < -125.0f) return 0.0f;
    float t = __fmaf_rn(-k, 0x1.62e430p-1f, x);
    t = __fmaf_rn(-k, -0x1.05c610p-29f, t);
    float q = 0x1.a01a02p-13f;
    q = __fmaf_rn(q, t, 0x1.6c16c2p-10f);
    q = __fmaf_rn(q, t, 0x1.111112p-7f);
    q = __fmaf_rn(q, t, 0x1.555556p-5f);
    q = __fmaf_rn(q, t, 0x1.555556p-3f);
    q = __fmaf_rn(q, t, 0.5f);
    q = __fmaf_rn(q, t, 1.0f);
    q = __fmaf_rn(q, t, 1.0f);
    return ldexpf(q, (int)k);
}

// The sampling distribution as exact integers: token v weighs E(v) =
// floor(exp_neg((z_v - max) / tau) 2^B), the argument by an fp32 subtraction
// and division (correctly rounded), B = 63 - ceil(log2(V + 1)) so that the
// row total S < 2^63; p(v) =
// E(v) / S.  Sums of weights are exact in any order, and the comparisons
// with a uniform U / 2^24 are exact 128-bit products, so the sampling
// decisions do not depend on how the work is split across threads.
__host__ __device__ __forceinline__ int sample_bits(int V)
{
    int b = 0;
    while ((1LL << b) < (long long)V + 1) b++;
    return 63 - b;
}

__device__ __forceinline__ unsigned long long weight_of(float z, float mx, float tau, int B)
{
    const float e = exp_neg(__fdiv_rn(__fsub_rn(z, mx), tau));
    return __float2ull_rz(ldexpf(e, B));
}

// Top-k order: token v of weight E ranks by the key E V + (V - 1 - v) (larger
// weight first, equal weights lower index first; distinct, < 2^63).  The
// top_k tokens are those whose key is at least the top_k-th largest key K
// (K = 0 keeps every token).
__device__ __forceinline__ unsigned long long top_key(unsigned long long E, int v, int V)
{
    return E * (unsigned long long)V + (unsigned long long)(V - 1 - v);
}

// The weight of token v in the restricted distribution.
__device__ __forceinline__ unsigned long long kept_weight(float z, int v, float mx, float tau, int B, int V,
                                                          unsigned long long K)
{
    const unsigned long long E = weight_of(z, mx, tau, B);
    return top_key(E, v, V) >= K ? E : 0ull;
}

// The top_k-th largest key of a row (all threads of the block): a radix
// select over the 64-bit keys, 8 bits per pass from the top; the keys are
// distinct, so after the last pass the prefix is that key.  Most keys share
// their high digits (most tokens have a tiny weight), so each warp counts
// equal digits once (one shared-memory atomic per distinct digit), and warp
// 0 finds the digit holding the wanted rank with a suffix scan over the 256
// buckets (8 per lane).  Once the keys still matching the prefix fit
// kTopCap, the next pass also gathers them into shared memory (s_keys, the
// caller's) and the passes after it read only those.  blockDim.x is a
// multiple of 32.
constexpr int kTopCap = 4096;

__device__ unsigned long long top_k_threshold(const float* __restrict__ z, int V, float mx, float tau, int B, int k,
                                              unsigned long long* s_keys)
{
    __shared__ unsigned int hist[256];
    __shared__ unsigned long long s_prefix;
    __shared__ unsigned int s_rank, s_sel, s_n;
    const int lane = threadIdx.x & 31;
    unsigned long long prefix = 0, mask = 0;
    int mode = 0;  // 0: every token; 1: every token, gathering the matching keys; 2: the gathered keys
    if (threadIdx.x == 0) s_rank = (unsigned int)k;  // rank among the keys that match the prefix (1 = largest)
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        if (threadIdx.x == 0 && mode == 1) s_n = 0;
        __syncthreads();
        const int n = mode == 2 ? (int)s_n : V, iters = (n + blockDim.x - 1) / blockDim.x;
        for (int it = 0; it < iters; it++) {
            const int i = it * blockDim.x + threadIdx.x;
            unsigned int d = 0xffffffffu;  // no bucket
            if (i < n) {
                const unsigned long long key = mode == 2 ? s_keys[i] : top_key(weight_of(z[i], mx, tau, B), i, V);
                if ((key & mask) == prefix) {
                    d = (unsigned int)(key >> shift) & 255u;
                    if (mode == 1) s_keys[atomicAdd(&s_n, 1u)] = key;
                }
            }
            const unsigned int peers = __match_any_sync(0xffffffffu, d);
            if (d != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (unsigned int)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l holds buckets 255-8l .. 248-8l (descending digit order)
            unsigned int c[8], part = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                c[j] = hist[255 - 8 * lane - j];
                part += c[j];
            }
            unsigned int incl = part;  // inclusive scan over lanes (higher digits first)
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned int rank = s_rank, before = incl - part;
            // the first lane whose buckets reach the rank picks the digit
            const unsigned int hit = __ballot_sync(0xffffffffu, incl >= rank);
            if (lane == __ffs(hit) - 1) {
                unsigned int cum = before;
                int d = 255 - 8 * lane - 7;  // the lowest digit of this lane, if the scan runs through
                for (int j = 0; j < 8; j++) {
                    if (cum + c[j] >= rank) {
                        d = 255 - 8 * lane - j;
                        break;
                    }
                    cum += c[j];
                }
                s_rank = rank - cum;
                s_sel = hist[d];  // keys matching the extended prefix
                s_prefix = prefix | ((unsigned long long)d << shift);
            }
        }
        __syncthreads();
        prefix = s_prefix;
        mask |= 255ull << shift;
        mode = mode == 1 ? 2 : (mode == 0 && s_sel <= (unsigned int)kTopCap ? 1 : mode);
        __syncthreads();
    }
    return prefix;
}

// a * b as 128 bits (hi, lo)
struct U128 {
    unsigned long long hi, lo;
};
__device__ __forceinline__ U128 mul128(unsigned long long a, unsigned long long b) { return {__umul64hi(a, b), a * b}; }
__device__ __forceinline__ U128 shl24(unsigned long long a) { return {a >> 40, a << 24}; }
__device__ __forceinline__ bool lt128(U128 a, U128 b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }

// Top-p bound after top-k (all threads of the block): among the tokens of
// key >= Kk (total weight Sk), in descending key order, the key of the first
// token whose running weight A reaches A 2^24 >= p24 Sk; *S_out = A.  The
// restriction keeps the keys >= the result, which is >= Kk.  A radix select
// like top_k_threshold's with each digit's weight in place of its count.
// When the active lanes of a warp share one digit (the first pass: most
// tokens have tiny weights), they add their weights with shuffles and one
// lane adds the total; otherwise each lane adds its own.  The buckets are
// 64-bit sums kept as two 32-bit words (the carry out of the low word goes
// to the high one), as 32-bit shared-memory atomics are native and 64-bit
// ones are not.  Only tokens of nonzero weight take part; the token found
// has nonzero weight.  Each pass keeps A_above (the weight of the keys above
// the prefix) with A_above 2^24 < p24 Sk <= (A_above + the prefix's weight)
// 2^24, so a digit reaching the bound always exists.
__device__ __forceinline__ void add_weight(unsigned int* lo, unsigned int* hi, unsigned long long w)
{
    const unsigned int l = (unsigned int)w, old = atomicAdd(lo, l);
    atomicAdd(hi, (unsigned int)(w >> 32) + (old + l < old ? 1u : 0u));
}

__device__ unsigned long long top_p_threshold(const float* __restrict__ z, int V, float mx, float tau, int B,
                                              unsigned long long Kk, unsigned long long Sk, unsigned int p24,
                                              unsigned long long* s_keys, unsigned long long* S_out)
{
    __shared__ unsigned int hlo[256], hhi[256], hc[256];
    __shared__ unsigned long long s_prefix, s_above, s_last;
    __shared__ unsigned int s_sel, s_n;
    const int lane = threadIdx.x & 31;
    const U128 target = mul128(p24, Sk);
    unsigned long long prefix = 0, mask = 0;
    int mode = 0;  // as in top_k_threshold
    if (threadIdx.x == 0) {
        s_above = 0;
        s_last = 0;
    }
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) {
            hlo[i] = 0;
            hhi[i] = 0;
            hc[i] = 0;
        }
        if (threadIdx.x == 0 && mode == 1) s_n = 0;
        __syncthreads();
        const int n = mode == 2 ? (int)s_n : V, iters = (n + blockDim.x - 1) / blockDim.x;
        for (int it = 0; it < iters; it++) {
            const int i = it * blockDim.x + threadIdx.x;
            unsigned int d = 0xffffffffu;  // no bucket
            unsigned long long w = 0;
            if (i < n) {
                unsigned long long key;
                if (mode == 2) {
                    key = s_keys[i];
                    w = key / (unsigned long long)V;
                } else {
                    w = weight_of(z[i], mx, tau, B);
                    key = top_key(w, i, V);
                }
                if (w != 0 && key >= Kk && (key & mask) == prefix) {
                    d = (unsigned int)(key >> shift) & 255u;
                    if (mode == 1) s_keys[atomicAdd(&s_n, 1u)] = key;
                } else {
                    w = 0;
                }
            }
            const unsigned int act = __ballot_sync(0xffffffffu, d != 0xffffffffu);
            if (act) {
                const unsigned int d0 = __shfl_sync(0xffffffffu, d, __ffs(act) - 1);
                if (__all_sync(0xffffffffu, d == d0 || d == 0xffffffffu)) {
                    unsigned long long t = w;  // the warp's total (< 2^63: part of one row's weight)
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    if (lane == 0) {
                        add_weight(&hlo[d0], &hhi[d0], t);
                        atomicAdd(&hc[d0], (unsigned int)__popc(act));
                    }
                } else if (d != 0xffffffffu) {
                    add_weight(&hlo[d], &hhi[d], w);
                    atomicAdd(&hc[d], 1u);
                }
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l holds buckets 255-8l .. 248-8l (descending digit order)
            unsigned long long c[8], part = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int b = 255 - 8 * lane - j;
                c[j] = ((unsigned long long)hhi[b] << 32) | hlo[b];
                part += c[j];
            }
            unsigned long long incl = part;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned long long above = s_above;
            const unsigned int hit = __ballot_sync(0xffffffffu, !lt128(shl24(above + incl), target));
            if (lane == (hit ? __ffs(hit) - 1 : 31)) {
                unsigned long long cum = above + incl - part;
                int d = 255 - 8 * lane - 7;
                for (int j = 0; j < 8; j++) {
                    if (!lt128(shl24(cum + c[j]), target)) {
                        d = 255 - 8 * lane - j;
                        break;
                    }
                    cum += c[j];
                }
                s_above = cum;
                s_last = ((unsigned long long)hhi[d] << 32) | hlo[d];
                s_sel = hc[d];
                s_prefix = prefix | ((unsigned long long)d << shift);
            }
        }
        __syncthreads();
        prefix = s_prefix;
        mask |= 255ull << shift;
        mode = mode == 1 ? 2 : (mode == 0 && s_sel <= (unsigned int)kTopCap ? 1 : mode);
        __syncthreads();
    }
    *S_out = s_above + s_last;
    return prefix;
}

// Uniform U: the top 24 bits of the next output (u = U / 2^24).
__device__ __forceinline__ unsigned long long uniform_u24(unsigned long long* x) { return smix64(x) >> 40; }

// Row max, threshold key K and total kept weight S for row 0 (block 0) and
// the verification rows vbase.. (blocks 1..): the rows whose softmax
// sampling verification reads.  stats[3r] = the max's float bits,
// stats[3r+1] = S, stats[3r+2] = K (0 without a top-k or top-p restriction;
// the kept tokens are those of key >= K).  p24 = floor(top_p 2^24), 2^24 for
// no top-p restriction.
constexpr int kStatThreads = 1024;  // one row per block: the selects' passes want every warp of an SM

__global__ void __launch_bounds__(kStatThreads) k_row_stats(const float* __restrict__ logits, int V, float tau,
                                                           int vbase, int T, int top_k, unsigned int p24,
                                                           unsigned long long* __restrict__ stats)
{
    __shared__ unsigned long long s_keys[kTopCap];  // the radix selects' gathered keys
    pdl_wait();
    pdl_trigger();
    // sequence blockIdx.y of a batch: its rows are T rows further on
    logits += (size_t)blockIdx.y * T * V;
    stats += (size_t)blockIdx.y * T * 3;
    const int r = blockIdx.x == 0 ? 0 : vbase + blockIdx.x - 1;
    const float* z = logits + (size_t)r * V;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, B = sample_bits(V);
    __shared__ float s_m[kStatThreads / 32];
    __shared__ unsigned long long s_s[kStatThreads / 32];
    float mx = -INFINITY;
    for (int v = threadIdx.x; v < V; v += kStatThreads) mx = fmaxf(mx, z[v]);
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_m[warp] = mx;
    __syncthreads();
    mx = s_m[0];
    for (int w = 1; w < kStatThreads / 32; w++) mx = fmaxf(mx, s_m[w]);
    unsigned long long K = (top_k > 0 && top_k < V) ? top_k_threshold(z, V, mx, tau, B, top_k, s_keys) : 0ull;
    unsigned long long sum = 0;
    for (int v = threadIdx.x; v < V; v += kStatThreads) sum += kept_weight(z[v], v, mx, tau, B, V, K);
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s_s[warp] = sum;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < kStatThreads / 32; w++) t += s_s[w];
    if (p24 < (1u << 24)) K = top_p_threshold(z, V, mx, tau, B, K, t, p24, s_keys, &t);
    if (threadIdx.x == 0) {
        stats[3 * r] = __float_as_uint(mx);
        stats[3 * r + 1] = t;
        stats[3 * r + 2] = K;
    }
}

void launch_row_stats(cudaStream_t s, const float* logits, int V, float tau, int vbase, int T,
                      unsigned long long* stats, int B, int top_k, unsigned int p24)
{
    launch_pdl(k_row_stats, dim3(1 + T - vbase, B), dim3(kStatThreads), 0, s, logits, V, tau, vbase, T, top_k,
               p24, stats);
}

// ------------------------------------------------- verify + harvest + shift ---

constexpr int kVerifyWarps = 32;  // window columns harvested at once (W <= kMaxW handled in rounds)

// Draw from the row's weights (max mx, total S) restricted to the tokens not
// in rej[0..nrej) (whose weight is R): the first token, in ascending order,
// whose running weight A has A 2^24 > U (S - R); the last admissible token of
// nonzero weight if none.  Every thread of the block takes part (a
// contiguous chunk of tokens each; chunk totals by a block scan, exact).
__device__ int block_draw(const float* z, int V, float tau, float mx, unsigned long long S, unsigned long long K,
                          const int* rej, int nrej, unsigned long long R, unsigned long long U)
{
    __shared__ unsigned long long s_part[kVerifyWarps];
    __shared__ int s_pick, s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x, B = sample_bits(V);
    const int chunk = (V + nt - 1) / nt, v0 = min(tid * chunk, V), v1 = min(v0 + chunk, V);
    const U128 target = mul128(U, S - R);
    auto weight = [&](int v) -> unsigned long long {
        for (int k = 0; k < nrej; k++)
            if (rej[k] == v) return 0ull;
        return kept_weight(z[v], v, mx, tau, B, V, K);
    };
    unsigned long long loc = 0;
    int last = -1;
    for (int v = v0; v < v1; v++) {
        const unsigned long long w = weight(v);
        loc += w;
        if (w) last = v;
    }
    unsigned long long x = loc;  // inclusive scan within the warp
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    if (tid == 0) {
        s_pick = INT_MAX;
        s_last = -1;
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long y = lane < nt / 32 ? s_part[lane] : 0ull;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += t;
        }
        s_part[lane] = y;
    }
    __syncthreads();
    const unsigned long long pre = (warp ? s_part[warp - 1] : 0ull) + x - loc;  // weight before this chunk
    if (last >= 0) atomicMax(&s_last, last);
    if (lt128(target, shl24(pre + loc))) {
        unsigned long long acc = pre;
        for (int v = v0; v < v1; v++) {
            acc += weight(v);
            if (lt128(target, shl24(acc))) {
                atomicMin(&s_pick, v);
                break;
            }
        }
    }
    __syncthreads();
    const int r = s_pick != INT_MAX ? s_pick : (s_last >= 0 ? s_last : 0);
    __syncthreads();
    return r;
}

// Sampling verification of one step (all threads of the block): writes the
// emitted tokens, committed rows and the advanced decode state, like the
// greedy branch of k_verify_update.
__device__ void sample_verify(DState* st, const int* tok, const float* logits, int V, float tau,
                              const unsigned long long* stats, int W, int N)
{
    __shared__ unsigned char s_alive[kRows];
    __shared__ int s_rej[kRows];
    __shared__ int s_nrej, s_acc, s_row, s_m, s_done, s_gbest, s_emit[kMaxN];
    __shared__ unsigned long long s_u, s_R;
    __shared__ unsigned long long s_rng;
    const int tid = threadIdx.x, n1 = N - 1, ncand = st->ncand, vbase = 1 + W * n1;
    if (tid == 0) {
        s_rng = st->rng;
        s_row = 0;
        s_m = 0;
        s_done = 0;
        s_gbest = -1;
    }
    for (int g = tid; g < kRows; g += blockDim.x) s_alive[g] = g < ncand;
    __syncthreads();
    for (int i = 0; i < n1; i++) {
        if (tid == 0) {
            const int row = s_row, B = sample_bits(V);
            const float* z = logits + (size_t)row * V;
            const float mx = __uint_as_float((unsigned)stats[3 * row]);
            const unsigned long long S = stats[3 * row + 1], K = stats[3 * row + 2];
            int nrej = 0, acc = -1;
            unsigned long long R = 0;
            for (int g = 0; g < ncand && acc < 0; g++) {
                if (!s_alive[g]) continue;
                const int v = tok[vbase + g * n1 + i];
                bool seen = false;
                for (int k = 0; k < nrej; k++) seen = seen || s_rej[k] == v;
                if (seen) continue;  // a value already tried at this level
                const unsigned long long U = uniform_u24(&s_rng), E = kept_weight(z[v], v, mx, tau, B, V, K);
                if (lt128(mul128(U, S - R), shl24(E))) {  // u (1 - R/S) < E/S
                    acc = g;
                } else {
                    s_rej[nrej++] = v;
                    R += E;
                }
            }
            s_acc = acc;
            s_nrej = nrej;
            s_R = R;
            if (acc < 0) s_u = uniform_u24(&s_rng);
        }
        __syncthreads();
        if (s_acc < 0) {
            const int row = s_row;
            const int v = block_draw(logits + (size_t)row * V, V, tau, __uint_as_float((unsigned)stats[3 * row]),
                                     stats[3 * row + 1], stats[3 * row + 2], s_rej, s_nrej, s_R, s_u);
            if (tid == 0) {
                s_emit[s_m] = v;
                s_done = 1;
            }
            __syncthreads();
            break;
        }
        if (tid == 0) {
            const int g = s_acc, v = tok[vbase + g * n1 + i];
            s_emit[s_m] = v;
            for (int h = 0; h < ncand; h++)
                if (s_alive[h] && tok[vbase + h * n1 + i] != v) s_alive[h] = 0;
            s_gbest = g;  // the lowest candidate still matching
            s_row = vbase + g * n1 + i;
            s_m = s_m + 1;
        }
        __syncthreads();
    }
    if (!s_done) {
        if (tid == 0) s_u = uniform_u24(&s_rng);
        __syncthreads();
        const int row = s_row;
        const int v = block_draw(logits + (size_t)row * V, V, tau, __uint_as_float((unsigned)stats[3 * row]),
                                 stats[3 * row + 1], stats[3 * row + 2], nullptr, 0, 0ull, s_u);
        if (tid == 0) s_emit[s_m] = v;
        __syncthreads();
    }
    if (tid == 0) {
        const int m = s_m, gs = s_gbest, P = st->P;
        for (int k = 0; k <= m; k++) st->emit[k] = s_emit[k];
        st->commit_rows[0] = 0;
        for (int k = 0; k < m; k++) st->commit_rows[k + 1] = vbase + gs * n1 + k;
        st->n_emit = m + 1;
        st->gstar = gs;
        st->P_before = P;
        st->P = P + m + 1;
        st->c = s_emit[m];
        st->steps += 1;
        st->rng = s_rng;
    }
}

// Verification, n-gram harvest and window shift of one step.
// Greedy verification (tau <= 0, warp 0): for each candidate g < G', m_g =
// the number of leading candidate tokens equal to the model's greedy choice
// at that point (the argmax of row 0 for the first, of row (g,i-1) for the
// i-th); the largest m wins, lowest g on ties; emit argmax(row 0) and the
// argmaxes of the m accepted rows.  Sampling verification (tau > 0, the
// whole block): sample_verify above.  Either way the decode state advances
// (P, c, emitted tokens, committed rows).  Harvest, from the window before
// the shift: warp j claims the slot of window column j's key; each key's
// lowest column then inserts that key's n-grams (win[1..N-2][j], argmax of
// row (N-2,j)) in ascending column order, so the pool holds what inserting
// columns 0..W-1 one after another gives (only the physical slot of
// colliding keys may differ, which lookups do not see).  Then every thread
// shifts the window up one level, the last level becoming the argmaxes of
// the last level's rows.
// Diagonal levels (diag): the n-gram keyed on win[0][j] steps one column
// right per level (win[l][j+l], then the argmax of row (N-2, j+N-2)), for
// the W-N+2 columns j whose diagonal stays inside the window; the new last
// level is the Jacobi update: argmax of row 0 in column 0, the argmax of the
// last level's row j-1 in column j.
__global__ void __launch_bounds__(kVerifyWarps * 32)
    k_verify_update(DState* st, const int* tok, const int* amax, int* win, PoolView pool, int W, int N, int G,
                    const float* logits, int V, float tau, const unsigned long long* stats, int diag,
                    const int* ovr, size_t sb)
{
    pdl_wait();
    pdl_trigger();
    {  // block b serves sequence b of a batch
        const int b = blockIdx.x;
        const size_t T = 1 + (size_t)(W + G) * (N - 1);
        st = seq_ptr(st, sb, b);
        win = seq_ptr(win, sb, b);
        pool = seq_pool(pool, sb, b);
        ovr = seq_ptr(ovr, sb, b);
        tok += b * T;
        amax += b * T;
        logits += b * T * V;
        stats += b * T * 3;
    }
    if (ovr[0]) amax = ovr + 1;  // debug: the rows' argmaxes set from the host
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n1 = N - 1, ncand = st->ncand, P = st->P;
    const int a0 = amax[0];
    const int vbase = 1 + W * n1;
    if (tau > 0.f) {
        sample_verify(st, tok, logits, V, tau, stats, W, N);
    } else if (warp == 0) {
        int best = -1;  // (m << 16) | (0xffff - g)
        for (int g0 = 0; g0 < ncand; g0 += 32) {
            int g = g0 + lane, key = -1;
            if (g < ncand) {
                int m = 0;
                while (m < n1) {
                    int expect = (m == 0) ? a0 : amax[vbase + g * n1 + m - 1];
                    if (tok[vbase + g * n1 + m] != expect) break;
                    m++;
                }
                key = (m << 16) | (0xffff - g);
            }
            for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
            best = max(best, key);
        }
        const int m = best < 0 ? 0 : (best >> 16);
        const int gs = best < 0 ? -1 : (0xffff - (best & 0xffff));
        if (lane == 0) {
            st->emit[0] = a0;
            st->commit_rows[0] = 0;
            for (int k = 0; k < m; k++) {
                st->emit[k + 1] = amax[vbase + gs * n1 + k];
                st->commit_rows[k + 1] = vbase + gs * n1 + k;
            }
            st->n_emit = m + 1;
            st->gstar = gs;
            st->P_before = P;
            st->P = P + m + 1;
            st->c = (m == 0) ? a0 : amax[vbase + gs * n1 + m - 1];
            st->steps += 1;
        }
    }
    // harvest from the window before the shift, in rounds of kVerifyWarps columns
    __shared__ int slot_of[kVerifyWarps];
    __shared__ int s_err;
    if (threadIdx.x == 0) s_err = 0;
    __syncthreads();
    const int n_grams = diag ? W - (n1 - 1) : W;  // keys win[0][0 .. n_grams)
    if (G > 0) {
        for (int j0 = 0; j0 < n_grams; j0 += kVerifyWarps) {
            const int j = j0 + warp;
            if (j < n_grams) {
                const int s = pool_claim(pool, win[j]);
                if (lane == 0) {
                    slot_of[warp] = s;
                    if (s < 0) s_err = 1;
                }
            }
            __syncthreads();
            if (!s_err && j < n_grams) {
                const int s = slot_of[warp];
                bool leader = true;
                for (int k = 0; k < warp; k++) leader = leader && slot_of[k] != s;
                if (leader) {
                    for (int jj = warp; jj < kVerifyWarps && j0 + jj < n_grams; jj++) {
                        if (slot_of[jj] != s) continue;
                        const int c = j0 + jj;
                        int val[kMaxN];
                        for (int l = 1; l < n1; l++) val[l - 1] = win[l * W + c + diag * l];
                        val[n1 - 1] = amax[1 + (n1 - 1) * W + c + diag * (n1 - 1)];
                        pool_insert_slot(pool, s, val);
                    }
                }
            }
            __syncthreads();
        }
        if (threadIdx.x == 0 && s_err) st->status = LA_ERR_CAPACITY;
    }
    __syncthreads();
    // window shift: level l <- level l+1; last level <- argmax of last level
    // rows (diagonal levels: of row 0, then of the last level's row j-1)
    const int nw = n1 * W, last0 = (n1 - 1) * W;
    int tmp[4];
    int k = 0;
    for (int idx = threadIdx.x; idx < nw; idx += blockDim.x)
        tmp[k++] = (idx < last0) ? win[idx + W] : (diag ? (idx == last0 ? a0 : amax[idx]) : amax[1 + idx]);
    __syncthreads();
    k = 0;
    for (int idx = threadIdx.x; idx < nw; idx += blockDim.x) win[idx] = tmp[k++];
}

void launch_verify_update(cudaStream_t s, DState* st, const int* tok, const int* amax, int* win, PoolView pool,
                          int W, int N, int G, const float* logits, int V, float tau,
                          const unsigned long long* stats, bool diag, const int* ovr, int B, size_t sb)
{
    launch_pdl(k_verify_update, dim3(B), dim3(kVerifyWarps * 32), 0, s, st, tok, amax, win, pool, W, N, G, logits,
               V, tau, stats, diag ? 1 : 0, ovr, sb);
}

// ------------------------------------------------------------------ commit ---

// Copy the step K/V of the committed rows into the cache for every layer:
// step layout [L][kRows][Hkv][hd], cache layout [L][Hkv][max_seq][hd].
// Step mode: rows st->commit_rows[0..n_emit) to positions P_before + i.
// Prefill mode: rows 0..n-1 to positions P + i.  Batched: grid z is the
// sequence, whose step rows start at row z * T.
__global__ void k_commit(const DState* st, int prefill, int n_prefill, const uint4* KS, const uint4* VS,
                         uint4* KC, uint4* VC, int Hkv, int hd_vec, int max_seq, int T, size_t sb)
{
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x, l = blockIdx.y, b = blockIdx.z;
    st = seq_ptr(st, sb, b);
    KC = seq_ptr(KC, sb, b);
    VC = seq_ptr(VC, sb, b);
    const int n = prefill ? n_prefill : st->n_emit;
    if (i >= n) return;
    const int row = (prefill ? i : st->commit_rows[i]) + b * T;
    const int p = (prefill ? st->P : st->P_before) + i;
    const int dkv_vec = Hkv * hd_vec;
    const size_t src = ((size_t)l * kRows + row) * dkv_vec;
    for (int e = threadIdx.x; e < dkv_vec; e += blockDim.x) {
        int h = e / hd_vec, x = e - h * hd_vec;
        size_t dst = (((size_t)l * Hkv + h) * max_seq + p) * hd_vec + x;
        KC[dst] = KS[src + e];
        VC[dst] = VS[src + e];
    }
}

void launch_commit(cudaStream_t s, const DState* st, bool prefill, int n_prefill, int n_max, const void* KS,
                   const void* VS, void* KC, void* VC, int L, int Hkv, int hd, int max_seq, int esz, int B, int T,
                   size_t sb)
{
    int hd_vec = hd * esz / 16;
    dim3 grid(prefill ? n_prefill : n_max, L, B);
    launch_pdl(k_commit, grid, dim3(256), 0, s, st, prefill ? 1 : 0, n_prefill, (const uint4*)KS, (const uint4*)VS,
               (uint4*)KC, (uint4*)VC, Hkv, hd_vec, max_seq, T, sb);
}

}  // namespace la

namespace la {

__global__ void k_set_state(DState* st, int P, int c, int reset)
{
    st->P = P;
    st->c = c;
    if (reset) {
        st->T = 0;
        st->ncand = 0;
        st->n_emit = 0;
        st->gstar = -1;
        st->P_before = P;
        st->status = 0;
        st->steps = 0;
    }
}

void launch_set_state(cudaStream_t s, DState* st, int P, int c, bool reset)
{
    k_set_state<<<1, 1, 0, s>>>(st, P, c, reset ? 1 : 0);
}

}  // namespace la
