// attn_tc.cu -- the decode step's masked attention on the Blackwell tensor
// cores (bf16, head_dim 64 or 128).
//
// Row r of a step, at position p = pos[r], attends to its visible sequence:
// the cache [0, P) and, at positions >= P, the step rows its row group sees
// (the combined 2D-window + verification mask of the lookahead step: the
// lookahead and verification branches of one forward pass, summary page,
// "Summary").  For lookahead output to equal greedy output bit for bit, the
// arithmetic of a row must depend on its own visible sequence only -- never
// on P, on the other rows of the step, or on where a key is read from.  So the
// keys of a row are split by the row's OWN position:
//
//   region A = [0, B(p)),  B(p) = 16 * floor((p - 31) / 16)  (0 for p < 31).
//     With the step's rows at most 31 positions past P (W + N - 2 <= 31),
//     B(p) <= P: region A is always in the cache.  It is processed in splits
//     of 128 absolute positions on tcgen05: per split, S = Q K^T
//     into tensor memory (M = 128 rows, N = 64 keys per MMA), one softmax
//     pass per row over the split's keys (max, exp2, sum in key order), the
//     probabilities in bf16 to shared memory, O = P V into tensor memory;
//     the split's (max, sum, O) goes to a partial buffer.  K and V stream in
//     by TMA (64-key boxes, 128-byte swizzle): K as the K-major B operand of
//     S, V as the MN-major B operand of O.
//   region B = [B(p), p]: the 32..47 most recent keys, the only keys where
//     rows of different groups differ.  Processed per row group on mma.sync
//     in 16-key tiles at absolute positions: each key row is
//     gathered (ldmatrix row addresses) from a TMA-staged cache window or
//     from the group's own step rows, so tile slot j always holds position
//     16t + j; online softmax across the tiles.
//
// A greedy row at the same position runs the same operations on the same
// values (same splits, same tiles, same instruction shapes); blocks and tiles
// that a step processes for other rows carry zero probabilities for it and
// add exact zeros.  Launch order: the cache kernel (region A; every CTA waits
// for the QKV epilogue before it triggers), then the window kernel (region B),
// which runs beside it -- it reads only data older than the cache kernel's
// wait -- then waits for it and merges: per row, M = the largest of the parts'
// maxima, O = the sum of exp2(m_part - M) O_part over region A's splits in
// ascending order and then region B (likewise the softmax sum), output
// O / sum in bf16.  The cache kernel's grid holds one CTA per (head group,
// split), sized by the caller to the splits the step needs (a smaller grid
// would have each CTA take splits blockIdx.y, + gridDim.y, ...).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>

#include "../../include/lookahead.h"
#include "common.cuh"
#include "ptx.cuh"

namespace la {

namespace {

using namespace ptx;

constexpr int kSA = 128;            // region-A split: absolute positions per partial state
constexpr int kBlk = 64;            // keys per TMA box / S MMA (N)
constexpr int kDelta = 31;          // region B: the keys within 31..46 positions of the row
constexpr int kAThreads = 320;      // warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 softmax / epilogue
constexpr uint32_t kTmemCols = 256; // S [128 columns] + O [head_dim columns]
constexpr int kBWarps = 8;          // region B: one row-group slab per warp
constexpr int kMaxSp = 32;          // region-A splits a row may have (max_seq <= 4096)

__host__ __device__ __forceinline__ int region_b_start(int p) { return p < kDelta ? 0 : ((p - kDelta) >> 4) << 4; }

__device__ __forceinline__ void raise_err(int* err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// Partial states: [H][nsa + 1][kRows][HD + 4] fp32 -- per (query head, part,
// row) the part's output sum O (HD values), its max and its softmax sum;
// parts 0..nsa-1 are region A's splits, part nsa is region B.
struct TcAttnArgs {
    const DState* st;
    RowSet rs;
    const int* pos;
    const __nv_bfloat16* Q;  // [rows][H * HD] (rotary embedding applied)
    __nv_bfloat16* out;      // [rows][H * HD]
    float* part;
    int* err;                // device status word (bounded waits)
    int rows, H, Hkv, max_seq, kv_row0;  // kv_row0: first cache-map row of this layer's KV head 0
    int ks_row0;             // first step-row-map row of this layer
    int max_rel;             // largest position offset of a step row
    int hpc, bq;             // region A: query heads per CTA, Q-tile rows per head
    int nsa;                 // region A: split slots
    float sl2;               // log2(e) / sqrt(head_dim)
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
__device__ __forceinline__ float* part_row(const TcAttnArgs& a, int h, int part, int r)
{
    return a.part + (((size_t)h * (a.nsa + 1) + part) * kRows + r) * (HD + 4);
}

// ------------------------------------------------------------ region A ---

template <int HD>
struct ASmem {
    static constexpr int kAtoms = HD / 64;                  // 128-byte atoms along head_dim
    static constexpr int kQ = 0;                             // Q [atom][128 rows][128 B]
    static constexpr int kQBytes = kAtoms * kRows * 128;
    static constexpr int kKBlock = kAtoms * kBlk * 128;      // one 64-key block of K or V
    static constexpr int kK = kQ + kQBytes;                  // K [block][atom][64 keys][128 B] ...
    static constexpr int kPBytes = 2 * kRows * 128;          // ... reused as P [atom of 64 keys][128 rows][128 B]
    static constexpr int kKBytes = 2 * kKBlock > kPBytes ? 2 * kKBlock : kPBytes;
    static constexpr int kV = kK + kKBytes;                  // V [block][atom][64 keys][128 B]
    // after a split's P.V, K/P and V (and a pad) stage the rows' partial
    // states [row][HD + 4] for one bulk store per head
    static constexpr int kStage = kK;
    static constexpr int kStageBytes = kRows * (HD + 4) * 4;
    static constexpr int kEnd0 = kV + 2 * kKBlock;
    static constexpr int kBar = kEnd0 > kStage + kStageBytes ? kEnd0 : kStage + kStageBytes;
    static constexpr int kRed = kBar + 128;  // the two column halves' max and sum per row [4][kRows]
    static constexpr int kBytes = kRed + 4 * kRows * 4;
};

template <int HD>
__global__ void __launch_bounds__(kAThreads, 2)
    k_attn_cache(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap, TcAttnArgs a)
{
    using L = ASmem<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bar = (uint64_t*)(sm + L::kBar);
    uint64_t *full_q = bar, *full_k = bar + 1, *full_v = bar + 2, *s_done = bar + 3, *p_ready = bar + 4,
             *o_done = bar + 5, *o_free = bar + 6;
    uint32_t* tmem_slot = (uint32_t*)(bar + 8);
    volatile int* abort_flag = (volatile int*)(bar + 9);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = blockIdx.x * a.hpc, kvh = h0 / (a.H / a.Hkv);
    const int kv_row = a.kv_row0 + kvh * a.max_seq;  // cache-map row of position 0 for this KV head

    // the cache (written by earlier steps) and P (set by the previous step's
    // verification) are older than every kernel of this step
    const int P = a.st->P;
    const int bmax = region_b_start(P + a.max_rel);
    const int nsp = (bmax + kSA - 1) / kSA;  // splits holding region-A keys of some row

    if (threadIdx.x == 0) {
        prefetch_map(&qmap);
        prefetch_map(&kmap);
        prefetch_map(&vmap);
        mbar_init(full_q, 1);
        mbar_init(full_k, 1);
        mbar_init(full_v, 1);
        mbar_init(s_done, 1);
        mbar_init(p_ready, 8);
        mbar_init(o_done, 1);
        mbar_init(o_free, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto split_blocks = [&](int sp) {
        const int lo = sp * kSA, hi = min(lo + kSA, bmax);
        return (hi - lo + kBlk - 1) / kBlk;
    };
    const uint64_t pol_kv = policy_evict_first();
    auto issue_kv = [&](int sp) {
        const int nb = split_blocks(sp), y0 = kv_row + sp * kSA;
        mbar_expect_tx(full_k, nb * L::kKBlock);
        for (int b = 0; b < nb; b++)
            for (int at = 0; at < L::kAtoms; at++)
                tma_load_2d(&kmap, full_k, sm + L::kK + b * L::kKBlock + at * (kBlk * 128), at * 64, y0 + b * kBlk,
                            pol_kv);
        mbar_expect_tx(full_v, nb * L::kKBlock);
        for (int b = 0; b < nb; b++)
            for (int at = 0; at < L::kAtoms; at++)
                tma_load_2d(&vmap, full_v, sm + L::kV + b * L::kKBlock + at * (kBlk * 128), at * 64, y0 + b * kBlk,
                            pol_kv);
    };
    // The first split's cached K and V were written by earlier steps: their
    // copies start before the wait.  Q is written by the QKV epilogue.  Every
    // CTA waits for it before it triggers: the window kernel launched next
    // relies on that for its reads.
    if (warp == 0 && lane == 0 && (int)blockIdx.y < nsp) issue_kv(blockIdx.y);
    pdl_wait();
    pdl_trigger();

    if ((int)blockIdx.y < nsp) {
        if (warp == 0) {
            if (lane == 0) {
                // ---------------- TMA producer
                const uint64_t pol_q = policy_evict_last();
                mbar_expect_tx(full_q, a.hpc * L::kAtoms * a.bq * 128);
                for (int hl = 0; hl < a.hpc; hl++)
                    for (int at = 0; at < L::kAtoms; at++)
                        tma_load_2d(&qmap, full_q, sm + L::kQ + at * (kRows * 128) + hl * a.bq * 128,
                                    (h0 + hl) * HD + at * 64, 0, pol_q);
                int n_kv = 1, it = 1;
                bool ok = true;
                for (int sp = blockIdx.y + gridDim.y; sp < nsp; sp += gridDim.y, it++) {
                    // K/P and V (the staging area too) are free once the
                    // previous split's partial states have been stored
                    if (!mbar_wait(o_free, (it - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    issue_kv(sp);
                    n_kv++;
                }
                if (!ok) {
                    *abort_flag = 1;
                    raise_err(a.err, LA_ERR_TIMEOUT);
                }
                // every copy issued lands before the CTA can exit
                mbar_drain(full_q, 0);
                mbar_drain(full_k, (n_kv - 1) & 1);
                mbar_drain(full_v, (n_kv - 1) & 1);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // ---------------- MMA issuer
                constexpr uint32_t id_s = idesc_bf16(128, kBlk, false);
                constexpr uint32_t id_o = idesc_bf16(128, HD, true);
                bool ok = mbar_wait(full_q, 0, abort_flag);
                int it = 0;
                for (int sp = blockIdx.y; sp < nsp && ok; sp += gridDim.y, it++) {
                    const int nb = split_blocks(sp);
                    const uint32_t par = it & 1;
                    if (!mbar_wait(full_k, par, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int b = 0; b < nb; b++)
#pragma unroll
                        for (int k = 0; k < HD / 16; k++) {
                            const uint32_t qa = smem_u32(sm + L::kQ + (k >> 2) * (kRows * 128)) + (k & 3) * 32;
                            const uint32_t ka =
                                smem_u32(sm + L::kK + b * L::kKBlock + (k >> 2) * (kBlk * 128)) + (k & 3) * 32;
                            mma_bf16(tmem + b * kBlk, desc_sw128_kmajor(qa), desc_sw128_kmajor(ka), id_s, k > 0);
                        }
                    mma_commit(s_done);
                    // O of the previous split must have been read before it is overwritten
                    if (!mbar_wait(p_ready, par, abort_flag) || !mbar_wait(full_v, par, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int b = 0; b < nb; b++)
#pragma unroll
                        for (int k = 0; k < kBlk / 16; k++) {
                            const uint32_t pa = smem_u32(sm + L::kK + b * (kRows * 128)) + k * 32;
                            const uint32_t va = smem_u32(sm + L::kV + b * L::kKBlock) + k * 16 * 128;
                            mma_bf16(tmem + 128, desc_sw128_kmajor(pa), desc_sw128_mnmajor(va, kBlk * 128), id_o,
                                     (b | k) != 0);
                        }
                    mma_commit(o_done);
                    // the next split's S may only be issued once its K has
                    // landed, which waits for o_free: S of split it+1 cannot
                    // overtake this split's softmax
                }
                if (!ok) {
                    *abort_flag = 1;
                    raise_err(a.err, LA_ERR_TIMEOUT);
                }
            }
        } else {
            // ---------------- softmax and epilogue: one thread per TMEM lane
            // (row) and column half -- two warps per lane quarter, one per
            // 64-key block of S and per half of O's columns
            const int q = warp & 3, v = q * 32 + lane, half = (warp - 2) >> 2;
            const int hl = v / a.bq, r = v - hl * a.bq;
            const bool valid = hl < a.hpc && r < a.rows;
            const int bnd = valid ? region_b_start(a.pos[r]) : 0;  // region A of this row: [0, bnd)
            const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
            float* srow = (float*)(sm + L::kStage) + (size_t)v * (HD + 4);
            float* red = (float*)(sm + L::kRed);  // [half] maxima, then [half] sums
            int it = 0;
            for (int sp = blockIdx.y; sp < nsp; sp += gridDim.y, it++) {
                const int nb = split_blocks(sp), lo = sp * kSA;
                const int nvis = min(max(bnd - lo, 0), nb * kBlk);
                const bool mine = half < nb;  // this warp's block holds keys (the same for the CTA)
                const uint32_t par = it & 1;
                if (!mbar_wait(s_done, par, abort_flag)) {
                    *abort_flag = 1;
                    raise_err(a.err, LA_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                // the row's max over its visible keys: each half's, then both
                float x[kBlk];
                float mh = -INFINITY;
                if (mine) {
                    tmem_ld64(trow + half * kBlk, x);
#pragma unroll
                    for (int j = 0; j < kBlk; j++)
                        if (half * kBlk + j < nvis) mh = fmaxf(mh, x[j] * a.sl2);
                }
                red[half * kRows + v] = mh;
                named_sync(1, 256);
                const float m = fmaxf(red[v], red[kRows + v]);
                const float mu = nvis > 0 ? m : 0.f;
                // probabilities and their sum in key order over this half's
                // keys, P in bf16 into its 128-byte-swizzled atom (the K-major
                // A operand of P.V); the row's sum is half 0's + half 1's
                float lh = 0.f;
                if (mine) {
#pragma unroll
                    for (int j = 0; j < kBlk; j++) {
                        const float pj = ex2(half * kBlk + j < nvis ? x[j] * a.sl2 - mu : -INFINITY);
                        x[j] = pj;
                        lh += pj;
                    }
                    uint8_t* prow = sm + L::kK + half * (kRows * 128) + v * 128;
#pragma unroll
                    for (int piece = 0; piece < 8; piece++) {
                        uint4 u;
                        u.x = pack2(x[piece * 8 + 0], x[piece * 8 + 1]);
                        u.y = pack2(x[piece * 8 + 2], x[piece * 8 + 3]);
                        u.z = pack2(x[piece * 8 + 4], x[piece * 8 + 5]);
                        u.w = pack2(x[piece * 8 + 6], x[piece * 8 + 7]);
                        *(uint4*)(prow + ((piece ^ (v & 7)) << 4)) = u;
                    }
                }
                red[(2 + half) * kRows + v] = lh;
                fence_proxy_async();  // P is read by the tensor core
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
                if (!mbar_wait(o_done, par, abort_flag)) {
                    *abort_flag = 1;
                    raise_err(a.err, LA_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                // this half of O's columns into the staging row (K/P and V are free now)
                constexpr int HC = HD / 2;
                if (HC == 64) {
                    tmem_ld64(trow + 128 + half * HC, x);
                } else {
                    tmem_ld32(trow + 128 + half * HC, x);
                }
#pragma unroll
                for (int j = 0; j < HC; j += 4)
                    *(float4*)(srow + half * HC + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                tc_fence_before();
                named_sync(1, 256);  // both halves' sums are in red
                if (half == 0) *(float2*)(srow + HD) = make_float2(m, red[2 * kRows + v] + red[3 * kRows + v]);
                fence_proxy_async();  // the staging rows are read by the bulk copy
                named_sync(1, 256);
                if (warp == 2 && lane == 0) {
                    // one bulk store of rows [0, rows) per query head of the CTA
                    for (int hh = 0; hh < a.hpc; hh++)
                        bulk_store(part_row<HD>(a, h0 + hh, sp, 0), sm + L::kStage + (size_t)hh * a.bq * (HD + 4) * 4,
                                   (uint32_t)a.rows * (HD + 4) * 4);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(o_free);
                }
            }
            if (warp == 2 && lane == 0) bulk_wait_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ region B ---

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
struct BSmem {
    static constexpr int kAtoms = HD / 64;
    static constexpr int kStep = kAtoms * kRows * 128;  // step K or V of one KV head [atom][128 rows][128 B]
    static constexpr int kWin = kAtoms * kBlk * 128;    // cache window K or V [atom][64 rows][128 B]
    // the staged K/V; after the tiles, the same bytes hold the merge's
    // per-slot region-B outputs [128 slots][HD + 4] and split weights [128][kMaxSp]
    static constexpr int kStageBytes = 2 * kStep + 2 * kWin;
    static constexpr int kMergeBytes = kRows * (HD + 4) * 4 + kRows * kMaxSp * 4;  // region-B outputs, split weights
    static constexpr int kArea = kStageBytes > kMergeBytes ? kStageBytes : kMergeBytes;
    static constexpr int kKS = 0;
    static constexpr int kVS = kKS + kStep;
    static constexpr int kKW = kVS + kStep;
    static constexpr int kVW = kKW + kWin;
    static constexpr int kZero = kArea;                 // one zero row (head_dim bf16)
    static constexpr int kBar = kZero + 256;
    static constexpr int kInts = kBar + 64;             // rows per group, slab prefix
    static constexpr int kSlot = kInts + ((2 * kRows + 2) * 4 + 15) / 16 * 16;  // per-slot merge state
    static constexpr int kBytes = kSlot + 7 * kRows * 4 + 16;
};

// The merge's arithmetic, spelled out as IEEE operations so that both merge
// paths below give a row the same bits: acc += x w per split in ascending
// order, and out = (acc + wB O_B) / sum, rounded to bf16.
__device__ __forceinline__ float4 fma4(float4 x, float w, float4 acc)
{
    return make_float4(__fmaf_rn(x.x, w, acc.x), __fmaf_rn(x.y, w, acc.y), __fmaf_rn(x.z, w, acc.z),
                       __fmaf_rn(x.w, w, acc.w));
}

__device__ __forceinline__ uint2 merge_out(float4 acc, float4 ob, float wB, float inv)
{
    const __nv_bfloat162 lo = __floats2bfloat162_rn(__fdiv_rn(__fmaf_rn(ob.x, wB, acc.x), inv),
                                                    __fdiv_rn(__fmaf_rn(ob.y, wB, acc.y), inv));
    const __nv_bfloat162 hi = __floats2bfloat162_rn(__fdiv_rn(__fmaf_rn(ob.z, wB, acc.z), inv),
                                                    __fdiv_rn(__fmaf_rn(ob.w, wB, acc.w), inv));
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    return u;
}

// The merge for CTAs holding a row with more than 8 region-A splits (long
// contexts): one thread per slot loads every split's (max, sum) together and
// puts the max, the splits' weights 2^(m - max) and the softmax sum (ascending
// split order, then region B) in shared memory; after a barrier the items
// (slot, 4 output dims; kIB per thread) load kSB splits' outputs at a time
// and sum them in ascending split order.  out = (O + wB O_B) / sum.
template <int HD>
__device__ void merge_long(const TcAttnArgs& a, int h, const float* sO, float* sW, const int* sRow, const int* sNA,
                           const float* sMB, const float* sLB, float* sWB, float* sLs, const int* sList,
                           int n_items, size_t pstride)
{
    constexpr int C4 = HD / 4, kIB = 2, kSB = 4;
    const int tid = threadIdx.x, dq = a.H * HD;
    if (tid < kRows && sRow[tid] >= 0) {
        const int slot = tid, nA = sNA[slot];
        const float* pr = part_row<HD>(a, h, 0, sRow[slot]) + HD;
        float2 ml[kMaxSp];
#pragma unroll
        for (int sp = 0; sp < kMaxSp; sp++)
            ml[sp] = sp < nA ? __ldcg((const float2*)(pr + sp * pstride)) : make_float2(-INFINITY, 0.f);
        float M = sMB[slot];
#pragma unroll
        for (int sp = 0; sp < kMaxSp; sp++) M = fmaxf(M, ml[sp].x);
        float Ls = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxSp; sp++) {
            if (sp < nA) {
                const float w = ex2(ml[sp].x - M);
                sW[slot * kMaxSp + sp] = w;
                Ls = __fmaf_rn(ml[sp].y, w, Ls);
            }
        }
        const float wB = ex2(sMB[slot] - M);
        sWB[slot] = wB;
        sLs[slot] = __fmaf_rn(sLB[slot], wB, Ls);
    }
    __syncthreads();
    for (int i0 = tid; i0 < n_items; i0 += kIB * blockDim.x) {
        int slot[kIB], nA[kIB];
        const float* pr[kIB];
        float4 acc[kIB];
        int nmax = 0;
#pragma unroll
        for (int k = 0; k < kIB; k++) {
            const int i = i0 + k * blockDim.x;
            slot[k] = i < n_items ? sList[i / C4] : 0;
            nA[k] = i < n_items ? sNA[slot[k]] : 0;
            pr[k] = part_row<HD>(a, h, 0, i < n_items ? sRow[slot[k]] : 0) + (i % C4) * 4;
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            nmax = max(nmax, nA[k]);
        }
        for (int s0 = 0; s0 < nmax; s0 += kSB) {
            float4 x[kIB][kSB];
#pragma unroll
            for (int k = 0; k < kIB; k++)
#pragma unroll
                for (int j = 0; j < kSB; j++)
                    x[k][j] = s0 + j < nA[k] ? __ldcg((const float4*)(pr[k] + (s0 + j) * pstride))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kIB; k++)
#pragma unroll
                for (int j = 0; j < kSB; j++) {
                    if (s0 + j < nA[k]) {
                        const float w = sW[slot[k] * kMaxSp + s0 + j];
                        acc[k] = fma4(x[k][j], w, acc[k]);
                    }
                }
        }
#pragma unroll
        for (int k = 0; k < kIB; k++) {
            const int i = i0 + k * blockDim.x;
            if (i >= n_items) continue;
            const int sl = slot[k], c4 = i % C4, r = sRow[sl];
            const float4 ob = *(const float4*)(sO + sl * (HD + 4) + c4 * 4);
            *(uint2*)(a.out + (size_t)r * dq + h * HD + c4 * 4) = merge_out(acc[k], ob, sWB[sl], sLs[sl]);
        }
    }
}

// at most 112 registers a thread: a window CTA (8 warps) then fits on an SM
// beside a cache CTA (10 warps at 96 registers) -- each of the SM's four
// register-file quarters holds 2 window warps next to up to 3 cache warps --
// so the two kernels overlap wherever the cache kernel's CTAs landed
template <int HD>
__global__ void __maxnreg__(112)
    k_attn_window(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ CUtensorMap ksmap, const __grid_constant__ CUtensorMap vsmap, TcAttnArgs a)
{
    using L = BSmem<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    uint64_t* full = (uint64_t*)(sm + L::kBar);
    volatile int* abort_flag = (volatile int*)(sm + L::kBar + 8);
    int* gcnt = (int*)(sm + L::kInts);  // [kRows + 1] rows of each group (< a.rows)
    int* gslab = gcnt + kRows + 1;      // [kRows + 1] slab prefix over groups
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, kvh = h / (a.H / a.Hkv);
    const int dq = a.H * HD;

    if (tid == 0) {
        mbar_init(full, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    // Everything read before pdl_wait() below is older than the cache
    // kernel's own wait: the cache, P, the rows' positions and tables, Q and
    // the step K/V written by the QKV epilogue.
    const int P = a.st->P;
    const int wstart = region_b_start(P);  // no row of the step sees a cached key before it
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = policy_evict_last();
        mbar_expect_tx(full, 2 * L::kStep + 2 * L::kWin);
        for (int at = 0; at < L::kAtoms; at++) {
            tma_load_2d(&ksmap, full, sm + L::kKS + at * (kRows * 128), kvh * HD + at * 64, a.ks_row0, pol);
            tma_load_2d(&vsmap, full, sm + L::kVS + at * (kRows * 128), kvh * HD + at * 64, a.ks_row0, pol);
            tma_load_2d(&kmap, full, sm + L::kKW + at * (kBlk * 128), at * 64, a.kv_row0 + kvh * a.max_seq + wstart,
                        pol);
            tma_load_2d(&vmap, full, sm + L::kVW + at * (kBlk * 128), at * 64, a.kv_row0 + kvh * a.max_seq + wstart,
                        pol);
        }
    }
    if (tid < 16) *(uint4*)(sm + L::kZero + tid * 16) = make_uint4(0, 0, 0, 0);
    const int ng = a.rs.ngrp;
    for (int g = tid; g < ng; g += blockDim.x) {
        int n = 0;
        for (int k = a.rs.grp_start[g]; k < a.rs.grp_start[g + 1]; k++) n += (a.rs.grp_rows[k] < a.rows);
        gcnt[g] = n;
    }
    __syncthreads();
    if (tid == 0) {
        gslab[0] = 0;
        for (int g = 0; g < ng; g++) gslab[g + 1] = gslab[g] + (gcnt[g] + 15) / 16;
    }
    __syncthreads();

    const int item = blockIdx.y * kBWarps + warp;
    const bool busy = item < gslab[ng];
    const int g4 = lane >> 2, t4 = lane & 3;
    int g = 0, rA = -1, rB = -1, posA = 0, posB = 0, bA = 0, bB = 0;
    uint32_t qf[HD / 16][4];
    if (busy) {
        while (gslab[g + 1] <= item) g++;
        const int* glist = a.rs.grp_rows + a.rs.grp_start[g];
        const int r_begin = (item - gslab[g]) * 16, r_end = gcnt[g];
        rA = (r_begin + g4 < r_end) ? glist[r_begin + g4] : -1;
        rB = (r_begin + g4 + 8 < r_end) ? glist[r_begin + g4 + 8] : -1;
        posA = rA >= 0 ? a.pos[rA] : -1;
        posB = rB >= 0 ? a.pos[rB] : -1;
        bA = rA >= 0 ? region_b_start(posA) : 0;
        bB = rB >= 0 ? region_b_start(posB) : 0;
        // Q fragments of the slab's rows (A operand) from global memory, while
        // the staging copies are in flight
        const __nv_bfloat16* qa = rA >= 0 ? a.Q + (size_t)rA * dq + h * HD : nullptr;
        const __nv_bfloat16* qb = rB >= 0 ? a.Q + (size_t)rB * dq + h * HD : nullptr;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ks++) {
            const int c0 = ks * 16 + 2 * t4;
            qf[ks][0] = qa ? *(const uint32_t*)(qa + c0) : 0u;
            qf[ks][1] = qb ? *(const uint32_t*)(qb + c0) : 0u;
            qf[ks][2] = qa ? *(const uint32_t*)(qa + c0 + 8) : 0u;
            qf[ks][3] = qb ? *(const uint32_t*)(qb + c0 + 8) : 0u;
        }
    }
    const bool staged = mbar_wait(full, 0, abort_flag);
    if (!staged) {
        raise_err(a.err, LA_ERR_TIMEOUT);
        mbar_drain(full, 0);
    }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[HD / 8][4];
#pragma unroll
    for (int d = 0; d < HD / 8; d++) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    if (busy && staged) {

    // the slab's tile range: union of its rows' windows (at most 4 tiles of 16)
    int lo = INT_MAX, hi = -1;
    if (rA >= 0) {
        lo = bA;
        hi = posA;
    }
    if (rB >= 0) {
        lo = min(lo, bB);
        hi = max(hi, posB);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    const int t0 = lo >> 4;
    int nt = (hi >> 4) - t0 + 1;  // warp-uniform
    if (nt > 4) {  // a step's row groups span at most 8 positions: never
        raise_err(a.err, LA_ERR_ARG);
        nt = 0;
    }
    const int* gmap = a.rs.grp_map + (size_t)g * a.rs.maxoff;
    const int kkey = (lane & 7) + ((lane >> 4) << 3);        // key row this lane addresses for K
    const int vkey = (lane & 7) + (((lane >> 3) & 1) << 3);  // ... and for V (transposed load)
    // Per tile, the K and V rows this lane addresses: the cache window, the
    // group's step row or the zero row, as (row base address, swizzle phase,
    // atom stride); chunk c of the row is then at base + (c / 8) * stride +
    // ((c % 8) ^ phase) * 16.
    uint32_t kb[4], vb[4], kst[4], vst[4];
    int ksw[4], vsw[4];
#pragma unroll
    for (int t = 0; t < 4; t++) {
#pragma unroll
        for (int role = 0; role < 2; role++) {
            const int p = (t0 + t) * 16 + (role ? vkey : kkey);
            uint32_t base = sb + L::kZero, stride = 0;
            int row = 0;
            if (t < nt) {
                if (p < P) {
                    row = p - wstart;
                    stride = kBlk * 128;
                    base = sb + (role ? L::kVW : L::kKW) + row * 128;
                } else if (p - P < a.rs.maxoff) {
                    row = gmap[p - P];
                    stride = kRows * 128;
                    base = sb + (role ? L::kVS : L::kKS) + row * 128;
                }
            }
            if (role) {
                vb[t] = base;
                vst[t] = stride;
                vsw[t] = stride ? (row & 7) : 0;
            } else {
                kb[t] = base;
                kst[t] = stride;
                ksw[t] = stride ? (row & 7) : 0;
            }
        }
    }
    auto chunk = [](uint32_t base, uint32_t stride, int sw, int c) {
        return base + (c >> 3) * stride + (((c & 7) ^ sw) << 4);
    };
    // S = Q K^T over the slab's tiles: two n8 tiles per 16-key tile, the
    // tiles' chains independent
    float s[4][2][4];
#pragma unroll
    for (int t = 0; t < 4; t++)
#pragma unroll
        for (int n = 0; n < 2; n++) s[t][n][0] = s[t][n][1] = s[t][n][2] = s[t][n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ks++) {
        const int c = 2 * ks + ((lane >> 3) & 1);
#pragma unroll
        for (int t = 0; t < 4; t++) {
            if (t < nt) {
                uint32_t b[4];
                ldsm_x4(b, chunk(kb[t], kst[t], ksw[t], c));
                mma16816(s[t][0], qf[ks], b[0], b[1]);
                mma16816(s[t][1], qf[ks], b[2], b[3]);
            }
        }
    }
    // one softmax pass per row over its window [B(p), p]: max, 2^(s - max),
    // sum in key order (this thread's keys ascending, then the 4 lanes of the
    // row in a fixed tree)
#pragma unroll
    for (int t = 0; t < 4; t++)
#pragma unroll
        for (int n = 0; n < 2; n++)
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int hh = i >> 1, kp = (t0 + t) * 16 + n * 8 + 2 * t4 + (i & 1);
                const bool vis = t < nt && (hh ? (rB >= 0 && kp >= bB && kp <= posB)
                                               : (rA >= 0 && kp >= bA && kp <= posA));
                const float x = vis ? s[t][n][i] * a.sl2 : -INFINITY;
                s[t][n][i] = x;
                m[hh] = fmaxf(m[hh], x);
            }
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
        m[hh] = fmaxf(m[hh], __shfl_xor_sync(0xffffffffu, m[hh], 1));
        m[hh] = fmaxf(m[hh], __shfl_xor_sync(0xffffffffu, m[hh], 2));
    }
    const float mu[2] = {m[0] == -INFINITY ? 0.f : m[0], m[1] == -INFINITY ? 0.f : m[1]};
    uint32_t pa[4][4];
#pragma unroll
    for (int t = 0; t < 4; t++) {
#pragma unroll
        for (int n = 0; n < 2; n++)
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float pv = ex2(s[t][n][i] - mu[i >> 1]);
                s[t][n][i] = pv;
                l[i >> 1] += pv;
            }
        pa[t][0] = pack_bf16(s[t][0][0], s[t][0][1]);
        pa[t][1] = pack_bf16(s[t][0][2], s[t][0][3]);
        pa[t][2] = pack_bf16(s[t][1][0], s[t][1][1]);
        pa[t][3] = pack_bf16(s[t][1][2], s[t][1][3]);
    }
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
    }
    // O = P V: one k16 step per tile, in tile order
#pragma unroll
    for (int t = 0; t < 4; t++) {
        if (t < nt) {
#pragma unroll
            for (int d2 = 0; d2 < HD / 16; d2++) {
                uint32_t b[4];
                ldsm_x4_t(b, chunk(vb[t], vst[t], vsw[t], 2 * d2 + (lane >> 4)));
                mma16816(o[2 * d2], pa[t], b[0], b[1]);
                mma16816(o[2 * d2 + 1], pa[t], b[2], b[3]);
            }
        }
    }
    }  // busy && staged

    // ---------------- merge with region A's splits (after the cache kernel) and write
    // Slot = warp * 16 + row of the warp's slab.  The staged K/V are dead once
    // every warp is past its tiles: their bytes take the slots' region-B
    // outputs and region A's split weights.
    float* sO = (float*)(sm + L::kKS);            // [slot][HD + 4]
    int* sRow = (int*)(sm + L::kSlot);            // row of the slot, -1 if none
    int* sNA = sRow + kRows;                      // region-A splits of the row
    float* sMB = (float*)(sNA + kRows);           // region B's max, sum and weight
    float* sLB = sMB + kRows;
    float* sWB = sLB + kRows;                     // long contexts: region B's weight and
    float* sLs = sWB + kRows;                     // the row's softmax sum over all parts
    float* sW = sO + kRows * (HD + 4);            // ... and the splits' weights [slot][kMaxSp]
    int* sList = (int*)(sLs + kRows);             // slots holding a row, their count, a long-context flag
    __syncthreads();
    if (busy && staged) {
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
            const int r = hh ? rB : rA, slot = warp * 16 + g4 + 8 * hh;
            if (t4 == 0) {
                sRow[slot] = r;
                sNA[slot] = r >= 0 ? ((hh ? bB : bA) + kSA - 1) / kSA : 0;
                sMB[slot] = m[hh];
                sLB[slot] = l[hh];
            }
            if (r >= 0) {
#pragma unroll
                for (int d = 0; d < HD / 8; d++)
                    *(float2*)(sO + slot * (HD + 4) + d * 8 + 2 * t4) = make_float2(o[d][2 * hh], o[d][2 * hh + 1]);
            }
        }
    } else if (lane < 16) {
        sRow[warp * 16 + lane] = -1;
    }
    constexpr int C4 = HD / 4, kIB = 2, kSB = 4, kMB = 8;
    if (tid == 0) {
        sList[kRows] = 0;
        sList[kRows + 1] = 0;
    }
    __syncthreads();
    // the slots holding a row (any order: it only assigns items to threads)
    if (tid < kRows && sRow[tid] >= 0) {
        sList[atomicAdd(&sList[kRows], 1)] = tid;
        if (sNA[tid] > kMB) sList[kRows + 1] = 1;
    }
    pdl_wait();  // the cache kernel is complete: its split partials are visible
    pdl_trigger();
    __syncthreads();
    const size_t pstride = (size_t)kRows * (HD + 4);  // from one split's partial to the next
    const int n_items = sList[kRows] * C4;
    if (sList[kRows + 1]) {
        merge_long<HD>(a, h, sO, sW, sRow, sNA, sMB, sLB, sWB, sLs, sList, n_items, pstride);
        return;
    }
    // Rows of at most kMB splits: per item (slot, 4 output dims; kIB per
    // thread at a time) the max over region B and every split, the splits'
    // weights 2^(m - max) and the softmax sum in ascending split order then
    // region B, and O = sum over splits (ascending) of w O_split + wB O_B;
    // out = O / sum.  Every split's (max, sum) and the first kSB splits'
    // outputs are loaded together: one round trip to L2 and no barrier.
    for (int i0 = tid; i0 < n_items; i0 += kIB * blockDim.x) {
        int slot[kIB], nA[kIB];
        const float *pr[kIB], *pm[kIB];
        int nmax = 0;
#pragma unroll
        for (int k = 0; k < kIB; k++) {
            const int i = i0 + k * blockDim.x;
            const bool ok = i < n_items;
            slot[k] = ok ? sList[i / C4] : 0;
            nA[k] = ok ? sNA[slot[k]] : 0;
            pm[k] = part_row<HD>(a, h, 0, ok ? sRow[slot[k]] : 0) + HD;
            pr[k] = pm[k] - HD + (i % C4) * 4;
            nmax = max(nmax, nA[k]);
        }
        float2 ml[kIB][kMB];
        float4 x[kIB][kSB];
#pragma unroll
        for (int k = 0; k < kIB; k++) {
#pragma unroll
            for (int j = 0; j < kMB; j++)
                ml[k][j] = j < nA[k] ? __ldcg((const float2*)(pm[k] + j * pstride)) : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int j = 0; j < kSB; j++)
                x[k][j] = j < nA[k] ? __ldcg((const float4*)(pr[k] + j * pstride)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float wB[kIB], inv[kIB], w[kIB][kMB];
        float4 acc[kIB];
#pragma unroll
        for (int k = 0; k < kIB; k++) {
            const bool ok = i0 + k * blockDim.x < n_items;
            float mx = ok ? sMB[slot[k]] : 0.f;
#pragma unroll
            for (int j = 0; j < kMB; j++) mx = fmaxf(mx, ml[k][j].x);
            float Ls = 0.f;
#pragma unroll
            for (int j = 0; j < kMB; j++) {
                w[k][j] = j < nA[k] ? ex2(ml[k][j].x - mx) : 0.f;
                if (j < nA[k]) Ls = __fmaf_rn(ml[k][j].y, w[k][j], Ls);
            }
            wB[k] = ok ? ex2(sMB[slot[k]] - mx) : 0.f;
            inv[k] = ok ? __fmaf_rn(sLB[slot[k]], wB[k], Ls) : 1.f;
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // splits 0 .. kMB-1: weights held in registers
#pragma unroll
        for (int c = 0; c < kMB / kSB; c++) {
            if (c * kSB >= nmax) break;
            if (c > 0) {
#pragma unroll
                for (int k = 0; k < kIB; k++)
#pragma unroll
                    for (int j = 0; j < kSB; j++)
                        x[k][j] = c * kSB + j < nA[k] ? __ldcg((const float4*)(pr[k] + (c * kSB + j) * pstride))
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < kIB; k++)
#pragma unroll
                for (int j = 0; j < kSB; j++) {
                    if (c * kSB + j < nA[k]) {
                        acc[k] = fma4(x[k][j], w[k][c * kSB + j], acc[k]);
                    }
                }
        }
#pragma unroll
        for (int k = 0; k < kIB; k++) {
            const int i = i0 + k * blockDim.x;
            if (i >= n_items) continue;
            const int sl = slot[k], c4 = i % C4, r = sRow[sl];
            const float4 ob = *(const float4*)(sO + sl * (HD + 4) + c4 * 4);
            *(uint2*)(a.out + (size_t)r * dq + h * HD + c4 * 4) = merge_out(acc[k], ob, wB[k], inv[k]);
        }
    }
}

// ------------------------------------------------------------------ host ---

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2D bf16 map over a row-major [rows][cols] matrix, box {64, box_rows},
// 128-byte swizzle; out-of-range rows read as zeros.
bool encode_map(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows)
{
    auto enc = encode_fn();
    if (!enc || !base || ((uintptr_t)base & 15) || (cols * 2) % 16) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int attn_tc_delta() { return kDelta; }

size_t attn_tc_partial_bytes(int H, int hd, int max_seq)
{
    const int nsa = (max_seq + kSA - 1) / kSA;
    return (size_t)H * (nsa + 1) * kRows * (hd + 4) * 4;
}

bool attn_tc_init(int hd)
{
    // both kernels prefer the largest shared-memory carveout, so that CTAs of
    // either fit beside the other's without reconfiguring an SM
    for (const void* f : {(const void*)k_attn_cache<128>, (const void*)k_attn_window<128>, (const void*)k_attn_cache<64>,
                          (const void*)k_attn_window<64>})
        if (cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) return false;
    if (hd == 128)
        return cudaFuncSetAttribute(k_attn_cache<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    ASmem<128>::kBytes + 1024) == cudaSuccess &&
               cudaFuncSetAttribute(k_attn_window<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    BSmem<128>::kBytes + 1024) == cudaSuccess;
    if (hd == 64)
        return cudaFuncSetAttribute(k_attn_cache<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    ASmem<64>::kBytes + 1024) == cudaSuccess &&
               cudaFuncSetAttribute(k_attn_window<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    BSmem<64>::kBytes + 1024) == cudaSuccess;
    return false;
}

const void* attn_tc_cache_kernel(int hd)
{
    return hd == 128 ? (const void*)k_attn_cache<128> : (const void*)k_attn_cache<64>;
}

int attn_tc_splits(const AttnTcPlan& pl, int P, int max_rel)
{
    const int nsp = (region_b_start(P + max_rel) + kSA - 1) / kSA;
    return nsp < 1 ? 1 : (nsp > pl.cta_cap ? pl.cta_cap : nsp);
}

int attn_tc_plan(AttnTcPlan* pl, const void* Q, int q_rows, const void* KC, const void* VC, long long kv_rows,
                 const void* KS, const void* VS, long long ks_rows, int H, int Hkv, int hd, int max_seq, int rows,
                 int n_items)
{
    memset(pl, 0, sizeof(*pl));
    if ((hd != 64 && hd != 128) || H % Hkv || rows < 1 || rows > kRows) return LA_ERR_ARG;
    // query heads per region-A CTA: heads of one KV head stacked as row blocks
    // of bq rows (a multiple of 8, so each block starts on a swizzle atom)
    int bq = 8;
    while (bq < rows) bq *= 2;
    int hpc = 1;
    const int group = H / Hkv;
    while (group % (2 * hpc) == 0 && 2 * hpc * bq <= kRows) hpc *= 2;
    const int nsa = (max_seq + kSA - 1) / kSA;
    if (nsa > kMaxSp) return LA_ERR_ARG;
    // one cache-kernel CTA per split: at long contexts its grid outgrows the
    // SMs' two slots per SM, and the window kernel's CTAs start as cache CTAs
    // leave; capping the grid so that both stay resident (each CTA taking
    // several splits in turn) was slower at the 13B and 34B contexts
    const int cap = nsa;
    const int dq = H * hd, dkv = Hkv * hd;
    if (!encode_map(&pl->qmap, Q, q_rows, dq, bq) || !encode_map(&pl->kmap, KC, kv_rows, hd, kBlk) ||
        !encode_map(&pl->vmap, VC, kv_rows, hd, kBlk) || !encode_map(&pl->ksmap, KS, ks_rows, dkv, kRows) ||
        !encode_map(&pl->vsmap, VS, ks_rows, dkv, kRows))
        return LA_ERR_CUDA;
    pl->H = H;
    pl->Hkv = Hkv;
    pl->hd = hd;
    pl->max_seq = max_seq;
    pl->hpc = hpc;
    pl->bq = bq;
    pl->nsa = nsa;
    pl->cta_cap = cap;
    pl->cache_smem = (hd == 128 ? ASmem<128>::kBytes : ASmem<64>::kBytes) + 1024;
    pl->n_items = n_items;
    pl->ok = true;
    return LA_OK;
}

void launch_attn_tc(cudaStream_t s, const AttnTcPlan& pl, int layer, int ks_row0, const DState* st, RowSet rs,
                    int max_rel, const int* pos, const void* Q, void* out, float* part, int rows, int* err, int cta_y)
{
    TcAttnArgs a{};
    a.st = st;
    a.rs = rs;
    a.pos = pos;
    a.Q = (const __nv_bfloat16*)Q;
    a.out = (__nv_bfloat16*)out;
    a.part = part;
    a.err = err;
    a.rows = rows;
    a.H = pl.H;
    a.Hkv = pl.Hkv;
    a.max_seq = pl.max_seq;
    a.kv_row0 = layer * pl.Hkv * pl.max_seq;
    a.ks_row0 = ks_row0;
    a.max_rel = max_rel;
    a.hpc = pl.hpc;
    a.bq = pl.bq;
    a.nsa = pl.nsa;
    a.sl2 = 1.4426950408889634f / sqrtf((float)pl.hd);
    const dim3 gc(pl.H / pl.hpc, cta_y < 1 ? 1 : cta_y), gw(pl.H, (pl.n_items + kBWarps - 1) / kBWarps);
    if (pl.hd == 128) {
        launch_pdl(k_attn_cache<128>, gc, dim3(kAThreads), pl.cache_smem, s, pl.qmap, pl.kmap, pl.vmap, a);
        launch_pdl(k_attn_window<128>, gw, dim3(kBWarps * 32), BSmem<128>::kBytes + 1024, s, pl.kmap, pl.vmap,
                   pl.ksmap, pl.vsmap, a);
    } else {
        launch_pdl(k_attn_cache<64>, gc, dim3(kAThreads), pl.cache_smem, s, pl.qmap, pl.kmap, pl.vmap, a);
        launch_pdl(k_attn_window<64>, gw, dim3(kBWarps * 32), BSmem<64>::kBytes + 1024, s, pl.kmap, pl.vmap,
                   pl.ksmap, pl.vsmap, a);
    }
}

}  // namespace la
