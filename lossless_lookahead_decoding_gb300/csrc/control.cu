// control.cu -- integer kernels of the lookahead step: row assembly with the
// pool lookup, greedy verification + n-gram harvest + window shift, KV commit,
// and the GPU n-gram pool (hash table) with warp-cooperative lookup/insert.
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
// insert index of each slot becomes that key's leader.
__global__ void k_pool_claim(PoolView p, const int* keys, int n)
{
    int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= n) return;
    int s = pool_claim(p, keys[w]);
    if ((threadIdx.x & 31) == 0) {
        p.slot_of[w] = s;
        if (s < 0) atomicExch(p.status, LA_ERR_CAPACITY);
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
    bool found;
    int s = pool_probe(p, keys[w], &found);
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
__global__ void k_build_rows(DState* st, const int* win, PoolView pool, int W, int N, int G, int T,
                             const int* rel_pos, int* tok, int* pos)
{
    __shared__ int s_slot, s_cnt;
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
    for (int r = threadIdx.x; r < kRows; r += blockDim.x) {
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
                       const int* rel_pos, int* tok, int* pos)
{
    k_build_rows<<<1, 128, 0, s>>>(st, win, pool, W, N, G, T, rel_pos, tok, pos);
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

// ------------------------------------------------- verify + harvest + shift ---

// One warp.  Verification: for each candidate g < G', m_g = number of leading
// candidate tokens equal to the model's greedy choice at that point (the
// argmax of row 0 for the first, of row (g,i-1) for the i-th); take the
// largest m, lowest g on ties; emit argmax(row 0) followed by the argmaxes of
// the m accepted rows.  Harvest: for j ascending insert key win[0][j] ->
// (win[1..N-2][j], argmax of row (N-2,j)).  Then shift the window up one
// level with those argmaxes as the new last level.  Finally advance P and c.
// Verification, n-gram harvest and window shift of one step.  Warp 0
// verifies (longest accepted prefix, lowest g on ties) and updates the decode
// state.  Harvest: warp j claims the slot of window column j's key; each key's
// lowest column then inserts that key's n-grams in ascending column order, so
// the pool holds what inserting columns 0..W-1 one after another gives (only
// the physical slot of colliding keys may differ, which lookups do not see).
// Then every thread shifts the window (after all harvest reads of it).
constexpr int kVerifyWarps = 32;  // window columns harvested at once (W <= kMaxW handled in rounds)

__global__ void __launch_bounds__(kVerifyWarps * 32) k_verify_update(DState* st, const int* tok, const int* amax,
                                                                     int* win, PoolView pool, int W, int N, int G)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n1 = N - 1, ncand = st->ncand, P = st->P;
    const int a0 = amax[0];
    const int vbase = 1 + W * n1;
    if (warp == 0) {
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
    if (G > 0) {
        for (int j0 = 0; j0 < W; j0 += kVerifyWarps) {
            const int j = j0 + warp;
            if (j < W) {
                const int s = pool_claim(pool, win[j]);
                if (lane == 0) {
                    slot_of[warp] = s;
                    if (s < 0) s_err = 1;
                }
            }
            __syncthreads();
            if (!s_err && j < W) {
                const int s = slot_of[warp];
                bool leader = true;
                for (int k = 0; k < warp; k++) leader = leader && slot_of[k] != s;
                if (leader) {
                    for (int jj = warp; jj < kVerifyWarps && j0 + jj < W; jj++) {
                        if (slot_of[jj] != s) continue;
                        const int c = j0 + jj;
                        int val[kMaxN];
                        for (int l = 1; l < n1; l++) val[l - 1] = win[l * W + c];
                        val[n1 - 1] = amax[1 + (n1 - 1) * W + c];
                        pool_insert_slot(pool, s, val);
                    }
                }
            }
            __syncthreads();
        }
        if (threadIdx.x == 0 && s_err) st->status = LA_ERR_CAPACITY;
    }
    __syncthreads();
    // window shift: level l <- level l+1; last level <- argmax of last level rows
    const int nw = n1 * W;
    int tmp[4];
    int k = 0;
    for (int idx = threadIdx.x; idx < nw; idx += blockDim.x) tmp[k++] = (idx < (n1 - 1) * W) ? win[idx + W] : amax[1 + idx];
    __syncthreads();
    k = 0;
    for (int idx = threadIdx.x; idx < nw; idx += blockDim.x) win[idx] = tmp[k++];
}

void launch_verify_update(cudaStream_t s, DState* st, const int* tok, const int* amax, int* win, PoolView pool,
                          int W, int N, int G)
{
    k_verify_update<<<1, kVerifyWarps * 32, 0, s>>>(st, tok, amax, win, pool, W, N, G);
}

// ------------------------------------------------------------------ commit ---

// Copy the step K/V of the committed rows into the cache for every layer:
// step layout [L][kRows][Hkv][hd], cache layout [L][Hkv][max_seq][hd].
// Step mode: rows st->commit_rows[0..n_emit) to positions P_before + i.
// Prefill mode: rows 0..n-1 to positions P + i.
__global__ void k_commit(const DState* st, int prefill, int n_prefill, const uint4* KS, const uint4* VS,
                         uint4* KC, uint4* VC, int Hkv, int hd_vec, int max_seq)
{
    const int i = blockIdx.x, l = blockIdx.y;
    const int n = prefill ? n_prefill : st->n_emit;
    if (i >= n) return;
    const int row = prefill ? i : st->commit_rows[i];
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
                   const void* VS, void* KC, void* VC, int L, int Hkv, int hd, int max_seq, int esz)
{
    int hd_vec = hd * esz / 16;
    dim3 grid(prefill ? n_prefill : n_max, L);
    k_commit<<<grid, 256, 0, s>>>(st, prefill ? 1 : 0, n_prefill, (const uint4*)KS, (const uint4*)VS, (uint4*)KC,
                                  (uint4*)VC, Hkv, hd_vec, max_seq);
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
