// gemm_tc.cu -- the bf16 decoder GEMMs on the 5th-generation tensor cores.
//
// One decode step multiplies <= 128 activation rows (the step's tokens) by
// every weight matrix once, so each GEMM streams its weights from HBM exactly
// once and is bound by HBM bandwidth.  Layout ("swap AB"): the weight matrix
// W [Nout][K] (row-major, K-major) is the 128-row A operand, the activations
// X [128][K] the N = 128 B operand, and the fp32 accumulator D[feature][token]
// lives in tensor memory.  Operands are staged into a 3-deep shared-memory
// ring of 128-K stages (two 64-K 128-byte-swizzle atoms per operand); one
// thread issues tcgen05.mma, one thread issues the copies, and four warps
// drain TMEM.
//
// Weight packing: at plan creation every weight matrix is copied once into
// "units" of 128 rows x 128 K, each stored as the exact shared-memory image
// the MMA reads (two 128-byte-swizzled 64-K atoms, zero padded past the
// matrix edge), units ordered tile-major then k.  A stage's weights are then
// one contiguous 32 KB bulk copy (cp.async.bulk) and a CTA's stream-K range
// is one contiguous stretch of HBM, instead of 128 scattered 256-byte row
// pieces per stage.  The activations stay row-major and come through a TMA
// tensor map (they are L2-resident and re-read by every CTA).
//
// Work split (stream-K): the flattened (tile, k-block) space is cut into
// equal contiguous ranges, one per CTA (one CTA per SM).  A CTA writes one
// fp32 partial per tile it touches; a second kernel sums the partials of a
// tile in ascending k order and applies the fused epilogue (RoPE, residual,
// SwiGLU, logits + argmax).  The split depends only on the matrix shape and
// the SM count, never on the number of rows, so every token's result is
// bit-identical whether it is decoded alone (greedy) or among 121 step rows
// (lookahead): this keeps lookahead output exactly the greedy output.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <initializer_list>
#include <utility>
#include <vector>

#include "gemm_tc.cuh"

namespace la {

namespace {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kBN = 128;                 // token columns (MMA N)
#ifndef LA_GEMM_ATOMS
#define LA_GEMM_ATOMS 2
#endif
constexpr int kAtom = 64;                // K per swizzle atom (one 128-byte row)
constexpr int kAtoms = LA_GEMM_ATOMS;    // atoms per pipeline stage
constexpr int kBK = kAtom * kAtoms;      // K per stage
#ifndef LA_GEMM_STAGES
#define LA_GEMM_STAGES 3
#endif
#ifndef LA_GEMM_CTAS_PER_SM
#define LA_GEMM_CTAS_PER_SM 1
#endif
constexpr int kStages = LA_GEMM_STAGES;
constexpr int kStageA = kBM * kBK * 2;   // 16 KB per atom
constexpr int kStageB = kBN * kBK * 2;   // 16 KB
constexpr int kThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTmemCols = 256;           // two 128-column fp32 accumulators
constexpr int kSmemBytes = kStages * (kStageA + kStageB) + 1024 + 256;
constexpr unsigned long long kWaitNs = 2000000000ull;  // bounded waits: 2 s

enum { EPI_LOGITS = 3 };

struct GemmArgs {
    int tiles, KB, ctas;
    int rows;        // tokens (columns) to store
    const uint8_t* wpack;  // packed weight units [tiles][KB] x kStageA bytes
    float* partial;  // [ctas + tiles][rows][128]
    int* err;        // device status word
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the given parity; gives up after kWaitNs or when
// another role has aborted.  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitNs) return false;
    }
}

// Contiguous global -> shared bulk copy (16-byte aligned, size a multiple of
// 16) completing on an mbarrier, with an L2 eviction-priority hint.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// TMA 2D tile load with an L2 eviction-priority hint (policy from
// createpolicy): weights are read once (evict first), activations are
// re-read by every CTA (evict last).
__device__ __forceinline__ void tma_load(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// K-major operand, 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                   // descriptor version
    d |= (uint64_t)2 << 61;                   // SWIZZLE_128B
    return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> f32, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N)
{
    return (1u << 4)                     // D format f32
           | (1u << 7)                   // A format bf16
           | (1u << 10)                  // B format bf16
           | ((uint32_t)(N >> 3) << 17)  // N / 8
           | ((uint32_t)(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__host__ __device__ __forceinline__ long long range_lo(int c, long long total, int ctas)
{
    return (long long)c * total / ctas;
}

__device__ __forceinline__ void raise_err(int* err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

__global__ void __launch_bounds__(kThreads, LA_GEMM_CTAS_PER_SM)
    k_gemm_tc(const __grid_constant__ CUtensorMap bmap, GemmArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kStageA;
    uint64_t* full = (uint64_t*)(sB + kStages * kStageB);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = (uint32_t*)(tempty + 2);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const long long total = (long long)g.tiles * g.KB;
    const long long lo = range_lo(c, total, g.ctas), hi = range_lo(c + 1, total, g.ctas);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; s++) issued[s] = false;
            bool ok = true;
            const uint64_t pw = policy_evict_first(), pa = policy_evict_last();
            auto load_a = [&](long long idx, int st) {
                bulk_load(sA + st * kStageA, g.wpack + (size_t)idx * kStageA, kStageA, &full[st], pw);
            };
            auto load_b = [&](long long idx, int st) {
#pragma unroll
                for (int a = 0; a < kAtoms; a++)
                    tma_load(&bmap, &full[st], sB + st * kStageB + a * (kBN * kAtom * 2),
                             (int)(idx % g.KB) * kBK + a * kAtom, 0, pa);
            };
            // The weights do not depend on the preceding kernels: fill the
            // ring with weight tiles before waiting for the activations the
            // predecessor writes (programmatic dependent launch).
            const int n_pre = (int)((hi - lo) < kStages ? (hi - lo) : kStages);
            for (int j = 0; j < n_pre; j++) {
                mbar_expect_tx(&full[j], kStageA + kStageB);
                load_a(lo + j, j);
                issued[j] = true;
                issued_phase[j] = 0;
            }
            pdl_wait();
            pdl_trigger();
            for (int j = 0; j < n_pre; j++) load_b(lo + j, j);
            stage = n_pre % kStages;
            phase = n_pre == kStages ? 1 : 0;
            for (long long idx = lo + n_pre; idx < hi; idx++) {
                if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&full[stage], kStageA + kStageB);
                load_a(idx, stage);
                load_b(idx, stage);
                issued[stage] = true;
                issued_phase[stage] = phase;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_err(g.err, LA_ERR_TIMEOUT);
                // let copies already in flight land before the CTA exits
                for (int s = 0; s < kStages; s++) {
                    if (!issued[s]) continue;
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&full[s], issued_phase[s]) && globaltimer() - t0 < kWaitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = make_idesc(kBM, kBN);
            int stage = 0, buf = 0, segs = 0;
            uint32_t phase = 0, tphase[2] = {0, 0};
            bool ok = true;
            for (long long idx = lo; idx < hi && ok; idx++) {
                const int kb = (int)(idx % g.KB);
                const bool first = (idx == lo) || kb == 0;
                const bool last = (idx == hi - 1) || kb == g.KB - 1;
                if (first && segs >= 2) {
                    if (!mbar_wait(&tempty[buf], tphase[buf], abort_flag)) {
                        ok = false;
                        break;
                    }
                    tphase[buf] ^= 1;
                    tc_fence_after();
                }
                if (!mbar_wait(&full[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(sA + stage * kStageA);
                const uint32_t b_base = smem_u32(sB + stage * kStageB);
                const uint32_t d = tmem + buf * kBN;
#pragma unroll
                for (int a = 0; a < kAtoms; a++)
#pragma unroll
                    for (int k = 0; k < kAtom / 16; k++)
                        mma_bf16(d, sw128_desc(a_base + a * (kBM * kAtom * 2) + k * 32),
                                 sw128_desc(b_base + a * (kBN * kAtom * 2) + k * 32), idesc,
                                 (first && a == 0 && k == 0) ? 0u : 1u);
                mma_commit(&empty[stage]);
                if (last) {
                    mma_commit(&tfull[buf]);
                    buf ^= 1;
                    segs++;
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_err(g.err, LA_ERR_TIMEOUT);
            }
        }
    } else {
        // ---------------- epilogue warps: TMEM -> fp32 partials
        pdl_wait();  // the partial buffer may still be read by the predecessor
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int buf = 0;
        uint32_t tphase[2] = {0, 0};
        if (lo < hi) {
            const int t_lo = (int)(lo / g.KB), t_hi = (int)((hi - 1) / g.KB);
            for (int t = t_lo; t <= t_hi; t++) {
                if (!mbar_wait(&tfull[buf], tphase[buf], abort_flag)) {
                    *abort_flag = 1;
                    raise_err(g.err, LA_ERR_TIMEOUT);
                    break;
                }
                tphase[buf] ^= 1;
                tc_fence_after();
                float* dst = g.partial + (size_t)(c + t) * g.rows * kBM + q * 32 + lane;
                for (int col0 = 0; col0 < g.rows; col0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * kBN + col0, v);
#pragma unroll
                    for (int j = 0; j < 32; j++)
                        if (col0 + j < g.rows) dst[(size_t)(col0 + j) * kBM] = v[j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                buf ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// Pack one weight matrix W [rows][K] (bf16, row-major) into units of the
// GEMM's ring: unit (t, kb) holds rows t*128.. and K columns kb*128.. as
// kAtoms 16 KB atoms; in an atom, 16-byte chunk c of row r (8 elements) sits
// at r*128 + ((c ^ (r & 7)) * 16), the 128-byte swizzle of the MMA operand
// descriptor.  Elements past the matrix edge are zero.  One thread per chunk.
__global__ void k_pack_sw128(const __nv_bfloat16* __restrict__ w, int rows, int K, int KB, int ntiles,
                             uint4* __restrict__ dst)
{
    const long long n = (long long)ntiles * KB * kAtoms * kBM * 8;
    const bool vec = (K % 8) == 0 && ((uintptr_t)w & 15) == 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(i & 7), r = (int)((i >> 3) & (kBM - 1));
        const long long atom = i >> 10;  // 8 chunks x 128 rows per atom
        const int a = (int)(atom % kAtoms);
        const long long unit = atom / kAtoms;
        const int kb = (int)(unit % KB), t = (int)(unit / KB);
        const int c = p ^ (r & 7);
        const int R = t * kBM + r, C = kb * kBK + a * kAtom + c * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (R < rows) {
            const __nv_bfloat16* src = w + (size_t)R * K + C;
            if (vec && C + 8 <= K) {
                v = *(const uint4*)src;
            } else {
                uint32_t u[4];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint32_t lo = C + 2 * j < K ? __bfloat16_as_ushort(src[2 * j]) : 0u;
                    const uint32_t hi = C + 2 * j + 1 < K ? __bfloat16_as_ushort(src[2 * j + 1]) : 0u;
                    u[j] = lo | (hi << 16);
                }
                v = make_uint4(u[0], u[1], u[2], u[3]);
            }
        }
        dst[i] = v;
    }
}

// ------------------------------------------------------------- epilogues ---

struct EpiArgs {
    int tiles, KB, ctas, rows, Nout;
    const float* __restrict__ partial;
    // QKV
    int dq, dkv, hd;
    const int* __restrict__ pos;
    const float* __restrict__ cosb;
    const float* __restrict__ sinb;
    __nv_bfloat16 *__restrict__ Q, *__restrict__ KS, *__restrict__ VS;
    // SwiGLU
    __nv_bfloat16* __restrict__ H;
    // logits / argmax
    float* __restrict__ logits;
    unsigned long long* amaxp;
};

struct ResidArgs {
    int tiles, KB, ctas, rows;
    const float* __restrict__ partial;
};

__device__ __forceinline__ int owner_cta(long long idx, long long total, int ctas)
{
    int c = (int)(idx * ctas / total);
    while (c > 0 && range_lo(c, total, ctas) > idx) c--;
    while (c + 1 < ctas && range_lo(c + 1, total, ctas) <= idx) c++;
    return c;
}

constexpr int kEpiRows = 8;

// Sum a tile's partials in ascending k order (all loads of a segment in
// flight together), then apply the fused epilogue for kEpiRows tokens.
template <int EPI>
__global__ void __launch_bounds__(128) k_gemm_epi(EpiArgs e)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, f = threadIdx.x;
    const long long total = (long long)e.tiles * e.KB;
    __shared__ float sbv[kEpiRows][4];
    __shared__ int sbi[kEpiRows][4];
    const int r0 = blockIdx.y * kEpiRows;
    // tile tt's partials for this thread's feature, rows r0.., ascending k
    // (the loads of two partials in flight together)
    auto sum_tile = [&](int tt, float* acc) {
        const int c_lo = owner_cta((long long)tt * e.KB, total, e.ctas);
        const int n = owner_cta((long long)tt * e.KB + e.KB - 1, total, e.ctas) - c_lo + 1;
        for (int q0 = 0; q0 < n; q0 += 2) {
            float v[2][kEpiRows];
#pragma unroll
            for (int q = 0; q < 2; q++)
#pragma unroll
                for (int i = 0; i < kEpiRows; i++) {
                    const int r = r0 + i;
                    v[q][i] = (q0 + q < n && r < e.rows) ? e.partial[((size_t)(c_lo + q0 + q + tt) * e.rows + r) * kBM + f]
                                                         : 0.f;
                }
#pragma unroll
            for (int q = 0; q < 2; q++)
                if (q0 + q < n) {
#pragma unroll
                    for (int i = 0; i < kEpiRows; i++) acc[i] = (q0 + q == 0) ? v[q][i] : acc[i] + v[q][i];
                }
        }
    };
    float acc[kEpiRows];
    sum_tile(t, acc);
    if (EPI == EPI_LOGITS) {
        const int fg = t * kBM + f;
        const bool valid = fg < e.Nout;
#pragma unroll
        for (int i = 0; i < kEpiRows; i++) {
            const int r = r0 + i;
            if (valid && e.logits && r < e.rows) e.logits[(size_t)r * e.Nout + fg] = acc[i];
            float bv = valid ? acc[i] : -INFINITY;
            int bi = valid ? fg : 0x7fffffff;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((f & 31) == 0) {
                sbv[i][f >> 5] = bv;
                sbi[i][f >> 5] = bi;
            }
        }
        __syncthreads();
        if (f < kEpiRows && r0 + f < e.rows) {
            float bv = sbv[f][0];
            int bi = sbi[f][0];
            for (int w = 1; w < 4; w++)
                if (sbv[f][w] > bv || (sbv[f][w] == bv && sbi[f][w] < bi)) {
                    bv = sbv[f][w];
                    bi = sbi[f][w];
                }
            if (bi != 0x7fffffff) {
                const uint32_t u = __float_as_uint(bv);
                const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                const unsigned long long packed = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)bi);
                atomicMax(&e.amaxp[r0 + f], packed);
            }
        }
    }
}

// Sum of stream-K partials for J (tile, feature) columns and R rows from
// r0: acc[j][i] = partials of tile tt[j], feature column f[j], row r0 + i,
// added in ascending k order; the loads of up to B partials of all columns
// are in flight together (a small B keeps registers low, so more epilogue
// CTAs are resident beside the GEMM they wait for).
constexpr int kSumBatch = 2;  // QKV epilogue

template <int J, int R, int B>
__device__ __forceinline__ void sum_partials(const EpiArgs& e, const int* tt, const int* f, int r0, float (*acc)[R])
{
    const long long total = (long long)e.tiles * e.KB;
    int lo[J], cnt[J], n = 0;
#pragma unroll
    for (int j = 0; j < J; j++) {
        lo[j] = owner_cta((long long)tt[j] * e.KB, total, e.ctas);
        cnt[j] = owner_cta((long long)tt[j] * e.KB + e.KB - 1, total, e.ctas) - lo[j] + 1;
        n = max(n, cnt[j]);
    }
    for (int q0 = 0; q0 < n; q0 += B) {
        float v[B][J][R];
#pragma unroll
        for (int q = 0; q < B; q++)
#pragma unroll
            for (int j = 0; j < J; j++)
#pragma unroll
                for (int i = 0; i < R; i++) {
                    const bool ok = q0 + q < cnt[j] && r0 + i < e.rows;
                    v[q][j][i] = ok ? e.partial[((size_t)(lo[j] + q0 + q + tt[j]) * e.rows + r0 + i) * kBM + f[j]] : 0.f;
                }
#pragma unroll
        for (int q = 0; q < B; q++)
#pragma unroll
            for (int j = 0; j < J; j++)
                if (q0 + q < cnt[j]) {
#pragma unroll
                    for (int i = 0; i < R; i++) acc[j][i] = (q0 + q == 0) ? v[q][j][i] : acc[j][i] + v[q][j][i];
                }
    }
}

// QKV epilogue: Q, K (rotate-half RoPE at each row's position) and V of the
// step rows, bf16.  Thread = (RoPE pair (fa, fa + hd/2) of the tile, R rows),
// a CTA 2R rows; the RoPE table entries do not depend on the GEMM and are
// fetched before waiting for it.  R = 8 for few rows; R = 11 for many (121
// rows: 576 CTAs of 128 registers a thread, one wave at 4 CTAs per SM, where
// R = 8 makes 768 CTAs of 96 registers and 5 per SM: 760 in the first wave).
template <int R>
__global__ void __launch_bounds__(128) k_epi_qkv(EpiArgs e)
{
    const int t = blockIdx.x, pr = threadIdx.x & 63;
    const int r0 = blockIdx.y * 2 * R + (threadIdx.x >> 6) * R;
    const int half = e.hd >> 1;
    const int fa = (pr / half) * e.hd + pr % half, fb = fa + half;
    const int ga = t * kBM + fa;
    const bool rope = ga < e.dq + e.dkv;
    float cs[R], sn[R];
#pragma unroll
    for (int i = 0; i < R; i++) {
        const int p = rope ? __ldcg(e.pos + min(r0 + i, e.rows - 1)) : 0;
        cs[i] = rope ? e.cosb[(size_t)p * half + pr % half] : 0.f;
        sn[i] = rope ? e.sinb[(size_t)p * half + pr % half] : 0.f;
    }
    pdl_wait();
    pdl_trigger();
    const int tt[2] = {t, t}, ff[2] = {fa, fb};
    float x[2][R];
    sum_partials<2, R, kSumBatch>(e, tt, ff, r0, x);
    if (rope) {
        const bool isq = ga < e.dq;
        __nv_bfloat16* dst = isq ? e.Q : e.KS;
        const int ld = isq ? e.dq : e.dkv, fl = isq ? ga : ga - e.dq;
#pragma unroll
        for (int i = 0; i < R; i++) {
            if (r0 + i < e.rows) {
                dst[(size_t)(r0 + i) * ld + fl] = __float2bfloat16_rn(x[0][i] * cs[i] - x[1][i] * sn[i]);
                dst[(size_t)(r0 + i) * ld + fl + half] = __float2bfloat16_rn(x[1][i] * cs[i] + x[0][i] * sn[i]);
            }
        }
    } else if (ga < e.dq + 2 * e.dkv) {
        const int fl = ga - e.dq - e.dkv;
#pragma unroll
        for (int i = 0; i < R; i++) {
            if (r0 + i < e.rows) {
                e.VS[(size_t)(r0 + i) * e.dkv + fl] = __float2bfloat16_rn(x[0][i]);
                e.VS[(size_t)(r0 + i) * e.dkv + fl + half] = __float2bfloat16_rn(x[1][i]);
            }
        }
    }
}

// SwiGLU epilogue: gate tiles come first, then the up tiles of the same
// features; H = silu(gate) * up in bf16.  Thread = (feature, ROWS rows), the
// loads of BATCH partials in flight at a time (the sums are the same for
// every ROWS and BATCH).  Few rows: ROWS = 8, BATCH = 2 (one round of loads).
// Many rows: ROWS = 16, BATCH = 1, at most 80 registers, so that the whole
// grid is resident beside the gate/up GEMM it waits for and, as it drains,
// still leaves room on every SM for the down GEMM's CTA to start fetching
// its weights.
template <int ROWS, int BATCH>
__global__ void __maxnreg__(80) k_epi_swiglu(EpiArgs e)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, f = threadIdx.x, r0 = blockIdx.y * ROWS;
    const int tt[2] = {t, t + e.tiles / 2}, ff[2] = {f, f};
    float x[2][ROWS];
    sum_partials<2, ROWS, BATCH>(e, tt, ff, r0, x);
    const int fo = t * kBM + f;
    if (fo < e.Nout) {
#pragma unroll
        for (int i = 0; i < ROWS; i++) {
            if (r0 + i < e.rows) {
                const float gt = x[0][i];
                e.H[(size_t)(r0 + i) * e.Nout + fo] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * x[1][i]);
            }
        }
    }
}

__global__ void k_argmax_unpack(unsigned long long* amaxp, int* amax, int rows)
{
    pdl_wait();
    pdl_trigger();
    const int r = threadIdx.x;
    if (r < rows) {
        amax[r] = (int)(0xFFFFFFFFu - (uint32_t)(amaxp[r] & 0xFFFFFFFFull));
        amaxp[r] = 0ull;
    }
}

// Residual add of a stream-K GEMM folded into the RMSNorm that follows it:
// per row, X += (the tile partials summed in ascending k order, as in every
// epilogue) then XN = X / sqrt(mean(X^2) + eps) * w in bf16.  One block of 1024 threads
// per row, VEC float4 per thread.
constexpr int kRnThreads = 1024, kRnSeg = 6;  // d <= VEC * 4 * 1024

template <int VEC>
__device__ __forceinline__ void resid_rmsnorm(const ResidArgs& a, float* __restrict__ X,
                                              const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ out,
                                              int d, float eps)
{
    const int r = blockIdx.x, d4 = d >> 2;
    float4* x = (float4*)(X + (size_t)r * d);
    const long long total = (long long)a.tiles * a.KB;
    __shared__ int s_lo[VEC * kRnThreads * 4 / kBM], s_n[VEC * kRnThreads * 4 / kBM];
    // Before the wait, what does not depend on the GEMM: the owner table, the
    // residual row and the norm weights.  The row's last writer (the previous
    // norm or the embedding) completed before the GEMM's CTAs passed their
    // own wait, and this kernel is launched only after all of them did.
    for (int t = threadIdx.x; t < a.tiles; t += kRnThreads) {
        const int lo = owner_cta((long long)t * a.KB, total, a.ctas);
        s_lo[t] = lo;
        s_n[t] = owner_cta((long long)t * a.KB + a.KB - 1, total, a.ctas) - lo + 1;
    }
    float4 v[VEC], wf[VEC];
#pragma unroll
    for (int i = 0; i < VEC; i++) {
        const int k = threadIdx.x + i * kRnThreads;
        if (k < d4) {
            v[i] = x[k];
            wf[i] = make_float4(__bfloat162float(w[4 * k]), __bfloat162float(w[4 * k + 1]),
                                __bfloat162float(w[4 * k + 2]), __bfloat162float(w[4 * k + 3]));
        } else {
            v[i] = wf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; i++) {
        const int k = threadIdx.x + i * kRnThreads;
        if (k >= d4) continue;
        const int t = (4 * k) / kBM, f = (4 * k) % kBM, lo = s_lo[t], n = s_n[t];
        const float4* src = (const float4*)&a.partial[((size_t)(lo + t) * a.rows + r) * kBM + f];
        const size_t seg = (size_t)a.rows * kBM / 4;  // float4 stride between segments
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < n; s0 += kRnSeg) {
            float4 p[kRnSeg];  // up to kRnSeg loads in flight, then summed in order
#pragma unroll
            for (int j = 0; j < kRnSeg; j++)
                p[j] = s0 + j < n ? __ldcg(src + (size_t)(s0 + j) * seg) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kRnSeg; j++) {
                if (s0 + j >= n) break;
                if (s0 + j == 0) {
                    acc = p[j];
                } else {
                    acc.x += p[j].x;
                    acc.y += p[j].y;
                    acc.z += p[j].z;
                    acc.w += p[j].w;
                }
            }
        }
        v[i] = make_float4(v[i].x + acc.x, v[i].y + acc.y, v[i].z + acc.z, v[i].w + acc.w);
        x[k] = v[i];
    }
#pragma unroll
    for (int i = 0; i < VEC; i++) {
        ss += v[i].x * v[i].x;
        ss += v[i].y * v[i].y;
        ss += v[i].z * v[i].z;
        ss += v[i].w * v[i].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float part[kRnThreads / 32];
    __shared__ float s_r;
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tt = 0.f;
        for (int i = 0; i < kRnThreads / 32; i++) tt += part[i];
        s_r = rsqrtf(tt / (float)d + eps);
    }
    __syncthreads();
    const float rr = s_r;
#pragma unroll
    for (int i = 0; i < VEC; i++) {
        const int k = threadIdx.x + i * kRnThreads;
        if (k < d4) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v[i].x * rr * wf[i].x, v[i].y * rr * wf[i].y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v[i].z * rr * wf[i].z, v[i].w * rr * wf[i].w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t*>(&lo);
            u.y = *reinterpret_cast<uint32_t*>(&hi);
            *(uint2*)(out + (size_t)r * d + 4 * k) = u;
        }
    }
}

// d <= 4096: at most 48 registers, so that the next GEMM's CTA (12 K
// registers) fits beside the norm's block and starts fetching its weights
// while the norm runs.
__global__ void __maxnreg__(48) k_resid_rmsnorm(ResidArgs a, float* __restrict__ X, const __nv_bfloat16* __restrict__ w,
                                                __nv_bfloat16* __restrict__ out, int d, float eps)
{
    resid_rmsnorm<1>(a, X, w, out, d, eps);
}

// 4096 < d <= 8192
__global__ void __launch_bounds__(kRnThreads) k_resid_rmsnorm_wide(ResidArgs a, float* __restrict__ X,
                                                                  const __nv_bfloat16* __restrict__ w,
                                                                  __nv_bfloat16* __restrict__ out, int d, float eps)
{
    resid_rmsnorm<2>(a, X, w, out, d, eps);
}


// ------------------------------------------------------------------ plan ---

struct GemmCfg {
    CUtensorMap b;
    int tiles, KB, ctas, Nout;
    size_t unit0;  // first packed unit of this GEMM
};

struct Impl {
    int sms = 0;
    int L = 0, d = 0, dq = 0, dkv = 0, hd = 0, F = 0, V = 0;
    std::vector<GemmCfg> qkv, oproj, gateup, down;
    GemmCfg lm;
    float* partial = nullptr;
    size_t partial_bytes = 0;
    uint8_t* wpack = nullptr;  // packed weight units of every GEMM
    size_t wpack_bytes = 0;
    int* err = nullptr;  // the context's device status word
    void* Q = nullptr;
    void* HID = nullptr;
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode()
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

// 2D bf16 tensor map over a row-major [rows][cols] matrix, box {64, box_rows}.
bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kAtom, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void finish_cfg(GemmCfg& g, int K, int sms)
{
    g.KB = (K + kBK - 1) / kBK;
    long long total = (long long)g.tiles * g.KB;
    const int slots = sms * LA_GEMM_CTAS_PER_SM;
    g.ctas = (int)(total < slots ? total : slots);
}

size_t partial_need(const GemmCfg& g) { return (size_t)(g.ctas + g.tiles) * kRows * kBM * 4; }

void launch_gemm(const TcPlan& p, const GemmCfg& g, cudaStream_t s, int rows, int cls)
{
    const Impl& im = *(const Impl*)p.impl;
    GemmArgs a{g.tiles, g.KB, g.ctas, rows, im.wpack + g.unit0 * kStageA, im.partial, im.err};
    if (p.prof) p.prof->begin(s);
    launch_pdl_carve(k_gemm_tc, dim3(g.ctas), dim3(kThreads), kSmemBytes, s, p.carveout, g.b, a);
    if (p.prof) {
        // algorithmic: every weight once, the rows' inputs once, the rows' outputs once
        const double K = (double)g.KB * kBK, Nw = (double)g.tiles * kBM;
        const double by = Nw * K * 2 + (double)rows * K * 2 + (double)rows * Nw * 2;
        p.prof->end(s, cls, by, 2.0 * rows * K * Nw);
    }
}

template <typename F>
void launch_epi(const TcPlan& p, cudaStream_t s, F f)
{
    if (p.prof) p.prof->begin(s);
    f();
    if (p.prof) p.prof->end(s, P_GEMM_EPI, 0, 0);
}

EpiArgs epi_base(const Impl& im, const GemmCfg& g, int rows)
{
    EpiArgs e{};
    e.tiles = g.tiles;
    e.KB = g.KB;
    e.ctas = g.ctas;
    e.rows = rows;
    e.Nout = g.Nout;
    e.partial = im.partial;
    return e;
}

dim3 epi_grid(const GemmCfg& g, int rows) { return dim3(g.tiles, (rows + kEpiRows - 1) / kEpiRows); }

}  // namespace

int tc_plan_create(TcPlan* p, const la_model_desc& d, const void* const* lw, void* XN, void* Q, void* ATT, void* HID,
                   int esz, int* status)
{
    p->ok = false;
    p->impl = nullptr;
    if (esz != 2) return 1;
    const int dq = d.n_heads * d.head_dim, dkv = d.n_kv_heads * d.head_dim;
    if (dq % kBM || dkv % kBM || d.d_model % kAtom || kBM % d.head_dim || d.head_dim % 2) return 1;
    if (d.d_model > 2 * 4 * kRnThreads) return 1;  // the residual norm's row limit
    if (!get_encode()) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (major < 10) return 1;
    Impl* im = new Impl();
    im->sms = sms;
    im->L = d.n_layers;
    im->d = d.d_model;
    im->dq = dq;
    im->dkv = dkv;
    im->hd = d.head_dim;
    im->F = d.ffn;
    im->V = d.vocab;
    im->Q = Q;
    im->HID = HID;
    bool ok = true;
    CUtensorMap bXN, bATT, bHID;
    ok &= make_map(&bXN, XN, kRows, d.d_model, kBN);
    ok &= make_map(&bATT, ATT, kRows, dq, kBN);
    ok &= make_map(&bHID, HID, kRows, d.ffn, kBN);
    // Packing jobs: (source matrix, its rows, K, first packed unit).
    struct PackJob {
        const void* w;
        int rows, K, KB, tiles;
        size_t unit0;
    };
    std::vector<PackJob> jobs;
    size_t units = 0;
    // A GEMM over the row-concatenation of up to three matrices [rows_i][K];
    // each matrix starts on a fresh 128-row tile.
    auto add_gemm = [&](GemmCfg& g, const CUtensorMap& b, int K, std::initializer_list<std::pair<const void*, int>> mats,
                        int Nout) {
        g.b = b;
        g.tiles = 0;
        g.Nout = Nout;
        g.KB = (K + kBK - 1) / kBK;
        g.unit0 = units;
        for (const auto& m : mats) {
            const int t = (m.second + kBM - 1) / kBM;
            jobs.push_back(PackJob{m.first, m.second, K, g.KB, t, units});
            units += (size_t)t * g.KB;
            g.tiles += t;
        }
        finish_cfg(g, K, sms);
    };
    size_t need = 0;
    for (int l = 0; l < d.n_layers && ok; l++) {
        const void* const* w = lw + (size_t)l * 9;
        GemmCfg q{}, o{}, gu{}, dn{};
        add_gemm(q, bXN, d.d_model, {{w[1], dq}, {w[2], dkv}, {w[3], dkv}}, dq + 2 * dkv);
        add_gemm(o, bATT, dq, {{w[4], d.d_model}}, d.d_model);
        add_gemm(gu, bXN, d.d_model, {{w[6], d.ffn}, {w[7], d.ffn}}, d.ffn);  // gate tiles, then up tiles
        add_gemm(dn, bHID, d.ffn, {{w[8], d.d_model}}, d.d_model);
        for (const GemmCfg* g : {&q, &o, &gu, &dn}) need = partial_need(*g) > need ? partial_need(*g) : need;
        im->qkv.push_back(q);
        im->oproj.push_back(o);
        im->gateup.push_back(gu);
        im->down.push_back(dn);
    }
    if (ok) {
        add_gemm(im->lm, bXN, d.d_model, {{d.lm_head, d.vocab}}, d.vocab);
        need = partial_need(im->lm) > need ? partial_need(im->lm) : need;
    }
    if (!ok) {
        delete im;
        return 1;
    }
    im->err = status;
    im->wpack_bytes = units * kStageA;
    if (cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess ||
        cudaMalloc((void**)&im->partial, need) != cudaSuccess ||
        cudaMalloc((void**)&im->wpack, im->wpack_bytes) != cudaSuccess) {
        if (im->partial) cudaFree(im->partial);
        delete im;
        return -1;
    }
    for (const PackJob& j : jobs) {
        const long long chunks = (long long)j.tiles * j.KB * kStageA / 16;
        const long long blocks = (chunks + 255) / 256;
        k_pack_sw128<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256>>>(
            (const __nv_bfloat16*)j.w, j.rows, j.K, j.KB, j.tiles, (uint4*)(im->wpack + j.unit0 * kStageA));
    }
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(im->partial);
        cudaFree(im->wpack);
        delete im;
        return -1;
    }
    im->partial_bytes = need;
    p->impl = im;
    p->ok = true;
    return 0;
}

void tc_plan_destroy(TcPlan* p)
{
    if (p->impl) {
        Impl* im = (Impl*)p->impl;
        if (im->partial) cudaFree(im->partial);
        if (im->wpack) cudaFree(im->wpack);
        delete im;
    }
    p->impl = nullptr;
    p->ok = false;
}

int* tc_status(const TcPlan& p) { return p.impl ? ((Impl*)p.impl)->err : nullptr; }

void tc_qkv_rope(const TcPlan& p, cudaStream_t s, int layer, int rows, const int* pos, const float* cosb,
                 const float* sinb, void* Q, void* KS, void* VS)
{
    const Impl& im = *(const Impl*)p.impl;
    const GemmCfg& g = im.qkv[layer];
    launch_gemm(p, g, s, rows, P_GEMM_QKV);
    EpiArgs e = epi_base(im, g, rows);
    e.dq = im.dq;
    e.dkv = im.dkv;
    e.hd = im.hd;
    e.pos = pos;
    e.cosb = cosb;
    e.sinb = sinb;
    e.Q = (__nv_bfloat16*)Q;
    e.KS = (__nv_bfloat16*)KS;
    e.VS = (__nv_bfloat16*)VS;
    launch_epi(p, s, [&] {
        if (rows <= 16)
            launch_pdl_carve(k_epi_qkv<8>, dim3(g.tiles, (rows + 15) / 16), dim3(128), 0, s, p.carveout, e);
        else
            launch_pdl_carve(k_epi_qkv<11>, dim3(g.tiles, (rows + 21) / 22), dim3(128), 0, s, p.carveout, e);
    });
}

TcResid tc_oproj(const TcPlan& p, cudaStream_t s, int layer, int rows)
{
    const Impl& im = *(const Impl*)p.impl;
    const GemmCfg& g = im.oproj[layer];
    launch_gemm(p, g, s, rows, P_GEMM_O);
    return TcResid{g.tiles, g.KB, g.ctas, rows, im.partial};
}

TcResid tc_down(const TcPlan& p, cudaStream_t s, int layer, int rows)
{
    const Impl& im = *(const Impl*)p.impl;
    const GemmCfg& g = im.down[layer];
    launch_gemm(p, g, s, rows, P_GEMM_DOWN);
    return TcResid{g.tiles, g.KB, g.ctas, rows, im.partial};
}

void tc_resid_rmsnorm(const TcPlan& p, cudaStream_t s, const TcResid& pend, float* X, const void* w, void* XN, int d,
                      float eps)
{
    ResidArgs a{pend.tiles, pend.KB, pend.ctas, pend.rows, pend.partial};
    if (p.prof) p.prof->begin(s);
    if (d <= 4 * kRnThreads)
        launch_pdl_carve(k_resid_rmsnorm, dim3(pend.rows), dim3(kRnThreads), 0, s, p.carveout, a, X,
                         (const __nv_bfloat16*)w, (__nv_bfloat16*)XN, d, eps);
    else
        launch_pdl_carve(k_resid_rmsnorm_wide, dim3(pend.rows), dim3(kRnThreads), 0, s, p.carveout, a, X,
                         (const __nv_bfloat16*)w, (__nv_bfloat16*)XN, d, eps);
    if (p.prof) p.prof->end(s, P_NORM, 0, 0);
}

void tc_gateup_swiglu(const TcPlan& p, cudaStream_t s, int layer, int rows)
{
    const Impl& im = *(const Impl*)p.impl;
    const GemmCfg& g = im.gateup[layer];
    launch_gemm(p, g, s, rows, P_GEMM_GU);
    EpiArgs e = epi_base(im, g, rows);
    e.H = (__nv_bfloat16*)im.HID;
    launch_epi(p, s, [&] {
        if (rows <= 16)
            launch_pdl_carve(k_epi_swiglu<8, 2>, dim3(g.tiles / 2, (rows + 7) / 8), dim3(128), 0, s, p.carveout, e);
        else
            launch_pdl_carve(k_epi_swiglu<16, 1>, dim3(g.tiles / 2, (rows + 15) / 16), dim3(128), 0, s, p.carveout,
                             e);
    });
}

void tc_lmhead_argmax(const TcPlan& p, cudaStream_t s, int rows, float* logits, unsigned long long* amaxp, int* amax)
{
    const Impl& im = *(const Impl*)p.impl;
    const GemmCfg& g = im.lm;
    launch_gemm(p, g, s, rows, P_GEMM_LM);
    EpiArgs e = epi_base(im, g, rows);
    e.logits = logits;
    e.amaxp = amaxp;
    launch_epi(p, s, [&] {
        launch_pdl_carve(k_gemm_epi<EPI_LOGITS>, epi_grid(g, rows), dim3(128), 0, s, p.carveout, e);
        launch_pdl_carve(k_argmax_unpack, dim3(1), dim3(kRows), 0, s, p.carveout, amaxp, amax, rows);
    });
}

}  // namespace la
