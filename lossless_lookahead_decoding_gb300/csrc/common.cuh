// common.cuh -- types shared by the kernels and the engine of liblookahead.so.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

constexpr int kRows = 128;   // rows of one forward pass (step rows or a prefill block)
constexpr int kMaxN = 8;     // largest n-gram size N
constexpr int kWarp = 32;

// Device-side decode state: read and written by the step's kernels so that a
// step is a fixed launch sequence (capturable in one CUDA graph).
struct DState {
    int P;         // tokens whose KV is in the cache
    int c;         // current token (its KV is not cached yet)
    int T;         // rows of the current step
    int ncand;     // candidates found in the pool for c (G')
    int n_emit;    // tokens emitted by the last step (m + 1)
    int gstar;     // chosen candidate, -1 if none
    int P_before;  // P at the start of the last step (commit base)
    int status;    // 0 or a negative LA_ERR_* raised on the device
    int emit[kMaxN];
    int commit_rows[kMaxN];
    long long steps;
    unsigned long long rng;  // sampling verification: splitmix64 stream state
};

// Static description of which in-step row provides the key at each position
// offset for every row group.  A row r of group grp[r] at position
// P + rel_pos[r] sees the cache [0,P) and, at offset o in [0, rel_pos[r]],
// the step row grp_map[grp[r]*maxoff + o].
struct RowSet {
    const int* rel_pos;
    const int* grp;
    const int* grp_map;
    const int* grp_start;  // [ngrp + 1] offsets into grp_rows
    const int* grp_rows;   // rows of each group in row order
    int maxoff;
    int ngrp;
};

// The n-gram pool: open-addressing hash table keyed on a token.  Each slot
// holds up to G (N-1)-grams, oldest first.
struct PoolView {
    int* keys;    // [cap], -1 = empty
    int* cnt;     // [cap]
    int* ent;     // [cap][G][n1]
    int* first;   // [cap] bulk-insert scratch (INT_MAX when idle)
    int* slot_of; // [max_bulk] bulk-insert scratch
    int* status;  // device int: set to LA_ERR_CAPACITY when full
    int cap;      // power of two
    int log2cap;
    int G, n1;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Batched decoding: the per-sequence state (KV cache, prompt, window, pool,
// decode state, argmax override) of sequence b sits b * sb bytes after
// sequence 0's; the sequences' step rows are consecutive T-row slices of the
// shared row arrays.  A kernel serving all sequences takes b from its grid.
template <typename P>
__host__ __device__ inline P* seq_ptr(P* p, size_t sb, int b)
{
    return reinterpret_cast<P*>(reinterpret_cast<uintptr_t>(p) + sb * (size_t)b);
}

__host__ __device__ inline PoolView seq_pool(PoolView p, size_t sb, int b)
{
    p.keys = seq_ptr(p.keys, sb, b);
    p.cnt = seq_ptr(p.cnt, sb, b);
    p.ent = seq_ptr(p.ent, sb, b);
    p.first = seq_ptr(p.first, sb, b);
    p.slot_of = seq_ptr(p.slot_of, sb, b);
    p.status = seq_ptr(p.status, sb, b);
    return p;
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- programmatic dependent launch (PDL) ----
// Kernels of the layer chain are launched with programmatic stream
// serialisation: a kernel may start while its predecessor drains.  Every such
// kernel calls pdl_wait() before touching data produced upstream (it returns
// once the predecessor grid has completed and its writes are visible) and
// then pdl_trigger() so that its own successor can be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// launch_pdl with a preferred shared-memory carveout (percent of the unified
// L1/shared array) for this launch; carveout < 0: the function's own setting.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_carve(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    int carveout, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    at[1].val.sharedMemCarveout = carveout < 0 ? 0u : (unsigned)carveout;
    cfg.attrs = at;
    cfg.numAttrs = carveout < 0 ? 1 : 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---- launchers (defined in the .cu files) ----
struct Dims {
    int L, d, H, Hkv, hd, F, V, max_seq;
    float eps;
};

// control.cu
void launch_build_rows(cudaStream_t s, DState* st, const int* win, PoolView pool, int W, int N, int G,
                       int T, const int* rel_pos, int* tok, int* pos, int B = 1, size_t sb = 0);
void launch_prefill_rows(cudaStream_t s, const DState* st, const int* prompt, int P0, int n, int* tok,
                         int* pos);
void launch_verify_update(cudaStream_t s, DState* st, const int* tok, const int* amax, int* win,
                          PoolView pool, int W, int N, int G, const float* logits, int V, float tau,
                          const unsigned long long* stats, bool diag, const int* ovr, int B = 1, size_t sb = 0);
void launch_row_stats(cudaStream_t s, const float* logits, int V, float tau, int vbase, int T,
                      unsigned long long* stats, int B = 1, int top_k = 0, unsigned int p24 = 1u << 24);
void launch_commit(cudaStream_t s, const DState* st, bool prefill, int n_prefill, int n_max, const void* KS,
                   const void* VS, void* KC, void* VC, int L, int Hkv, int hd, int max_seq, int esz, int B = 1,
                   int T = 0, size_t sb = 0);
void launch_pool_reset(cudaStream_t s, PoolView pool);
void launch_set_state(cudaStream_t s, DState* st, int P, int c, bool reset);
void launch_pool_insert(cudaStream_t s, PoolView pool, const int* keys, const int* grams, int gram_stride,
                        int n);
void launch_pool_lookup(cudaStream_t s, PoolView pool, const int* keys, int n, int* out, int* counts);

// simt.cu (T = element type of weights/activations: float or bf16)
template <typename T>
void launch_embed(cudaStream_t s, const int* tok, const T* emb, float* X, int rows, int d);
template <typename T>
void launch_rmsnorm(cudaStream_t s, const float* X, const T* w, T* out, int rows, int d, float eps);
template <typename T>
void launch_gemm_simt_f32out(cudaStream_t s, const T* A, const T* W, float* out, int ld_out, int rows, int K,
                             int Nout);
template <typename T>
void launch_gemm_simt_resid(cudaStream_t s, const T* A, const T* W, float* X, int rows, int K, int Nout);
template <typename T>
void launch_gemm_simt_swiglu(cudaStream_t s, const T* A, const T* Wg, const T* Wu, T* out, int rows, int K,
                             int F);
template <typename T>
void launch_rope_split(cudaStream_t s, const float* qkv, const int* pos, const float* cosb, const float* sinb,
                       T* Q, T* KS, T* VS, int rows, int H, int Hkv, int hd);
template <typename T>
void launch_attn_simt(cudaStream_t s, const DState* st, RowSet rs, const int* pos, const T* Q, const T* KC,
                      const T* VC, const T* KS, const T* VS, T* out, int rows, int H, int Hkv, int hd,
                      int max_seq, float scale);
void launch_argmax(cudaStream_t s, const float* logits, int* amax, int rows, int V);

// attn_tc.cu (bf16, head_dim 64 or 128): the decode step's attention on
// tcgen05 (cached keys older than the row's recent window) + mma.sync (the
// recent window, per row group), merged per row
struct AttnTcPlan {
    CUtensorMap qmap, kmap, vmap, ksmap, vsmap;
    int H, Hkv, hd, max_seq, hpc, bq, nsa, cta_cap, n_items, cache_smem;
    bool ok;
};
int attn_tc_delta();  // rows may sit at most this many positions past P
size_t attn_tc_partial_bytes(int H, int hd, int max_seq);
bool attn_tc_init(int hd);
// Q: [q_rows][H*hd]; KC/VC: [kv_rows][hd] (layers x KV heads x max_seq rows);
// KS/VS: [ks_rows][Hkv*hd] (step rows of every layer); n_items: row-group
// slabs of 16 rows of the step's row table
int attn_tc_plan(AttnTcPlan* pl, const void* Q, int q_rows, const void* KC, const void* VC, long long kv_rows,
                 const void* KS, const void* VS, long long ks_rows, int H, int Hkv, int hd, int max_seq, int rows,
                 int n_items);
// cta_y: region-A CTAs per head group (the cache kernel's grid.y), from
// attn_tc_splits() for the step's P; attn_tc_cache_kernel() identifies that
// kernel's launches in a captured graph, whose grids the caller updates when
// the split count changes
void launch_attn_tc(cudaStream_t s, const AttnTcPlan& pl, int layer, int ks_row0, const DState* st, RowSet rs,
                    int max_rel, const int* pos, const void* Q, void* out, float* part, int rows, int* err, int cta_y);
int attn_tc_splits(const AttnTcPlan& pl, int P, int max_rel);
const void* attn_tc_cache_kernel(int hd);

// attn_mma.cu (bf16, head_dim 64 or 128): prefill blocks (causal)
size_t attn_mma_partial_bytes(int H, int hd, int max_seq);
bool attn_mma_init(int hd);
void launch_attn_mma(cudaStream_t s, const DState* st, RowSet rs, int max_rel, const int* pos, const void* Q,
                     const void* KC, const void* VC, const void* KS, const void* VS, void* out, float* part, int rows,
                     int H, int Hkv, int hd, int max_seq, int B = 1, size_t sb = 0);

}  // namespace la

#include <vector>

namespace la {

// Optional per-kernel-class timing: CUDA event pairs recorded on the launching
// stream around each instrumented launch (also inside a captured graph).
enum ProfClass {
    P_GEMM_QKV = 0, P_GEMM_O, P_GEMM_GU, P_GEMM_DOWN, P_GEMM_LM, P_GEMM_EPI, P_ATTN, P_NORM, P_CONTROL, P_NCLS
};

struct ProfPoint {
    int cls;
    double bytes, flops;  // algorithmic per launch (attention: filled per step)
    cudaEvent_t a, b;
};

struct Profiler {
    bool on = false;
    std::vector<ProfPoint> pts;
    size_t idx = 0;
    double ms[P_NCLS] = {}, bytes[P_NCLS] = {}, flops[P_NCLS] = {};
    long long n[P_NCLS] = {};
    void begin(cudaStream_t s)
    {
        if (!on) return;
        if (idx == pts.size()) {
            ProfPoint p{};
            cudaEventCreate(&p.a);
            cudaEventCreate(&p.b);
            pts.push_back(p);
        }
        cudaEventRecord(pts[idx].a, s);
    }
    void end(cudaStream_t s, int cls, double by, double fl)
    {
        if (!on) return;
        ProfPoint& p = pts[idx++];
        p.cls = cls;
        p.bytes = by;
        p.flops = fl;
        cudaEventRecord(p.b, s);
    }
    ~Profiler()
    {
        for (auto& p : pts) {
            cudaEventDestroy(p.a);
            cudaEventDestroy(p.b);
        }
    }
};

}  // namespace la
