// simt.cu -- CUDA-core kernels of the decoder forward: embedding gather,
// RMSNorm, SIMT GEMMs (fp32 debug path and fallback), RoPE, the masked
// lookahead/verification attention, and the per-row argmax.
//
// Every kernel computes each row's result as a function of that row's inputs
// only, with a reduction order that does not depend on how many rows the
// launch holds.  The attention walks keys in chunks aligned to absolute
// positions (multiples of 32) in ascending order.  Together these make a
// token's logits in a lookahead step bit-identical to the same token's logits
// in plain greedy decoding, which is what keeps the decoded output exactly
// the greedy output (summary page of Fu et al. 2024, "Summary").
#include "common.cuh"

namespace la {

// ---------------------------------------------------------------- embed ---
// One block per row; 16-byte loads of the embedding row (all of a thread's
// loads in flight together) when d and the table allow, else one element at
// a time.
constexpr int kEmbVec = 4;  // 16-byte loads per thread: d <= 4 * 256 * (16 / sizeof(T))

template <typename T>
__global__ void k_embed(const int* tok, const T* emb, float* X, int d)
{
    pdl_wait();
    pdl_trigger();
    constexpr int E = 16 / sizeof(T);  // elements per 16-byte load
    const int r = blockIdx.x;
    const T* e = emb + (size_t)tok[r] * d;
    float* x = X + (size_t)r * d;
    if (d % E == 0 && d <= kEmbVec * E * (int)blockDim.x && ((uintptr_t)emb & 15) == 0) {
        uint4 v[kEmbVec];
#pragma unroll
        for (int i = 0; i < kEmbVec; i++) {
            const int k = (threadIdx.x + i * blockDim.x) * E;
            v[i] = k < d ? *(const uint4*)(e + k) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kEmbVec; i++) {
            const int k = (threadIdx.x + i * blockDim.x) * E;
            if (k >= d) continue;
            const T* t = reinterpret_cast<const T*>(&v[i]);
#pragma unroll
            for (int j = 0; j < E; j += 4) *(float4*)(x + k + j) = make_float4(to_f(t[j]), to_f(t[j + 1]), to_f(t[j + 2]), to_f(t[j + 3]));
        }
        return;
    }
    for (int k = threadIdx.x; k < d; k += blockDim.x) x[k] = to_f(e[k]);
}

template <typename T>
void launch_embed(cudaStream_t s, const int* tok, const T* emb, float* X, int rows, int d)
{
    launch_pdl(k_embed<T>, dim3(rows), dim3(256), 0, s, tok, emb, X, d);
}

// -------------------------------------------------------------- rmsnorm ---
// x / sqrt(mean(x^2) + eps) * w  (Zhang and Sennrich 2019, cited by the
// pages).  One block per row; each thread loads its float4 slices up front
// (all loads in flight at once), sums squares in a fixed order, then a fixed
// xor tree and the warps in order.
constexpr int kNormThreads = 256, kNormVec = 8;  // d <= 8 * 4 * 256 = 8192

__device__ __forceinline__ void store4(float* o, float a, float b, float c, float d)
{
    *(float4*)o = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(__nv_bfloat16* o, float a, float b, float c, float d)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *(uint2*)o = u;
}

template <typename T>
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const float* X, const T* w, T* out, int d, float eps)
{
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x, d4 = d >> 2;
    const float4* x = (const float4*)(X + (size_t)r * d);
    float4 v[kNormVec];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormVec; i++) {
        const int k = threadIdx.x + i * kNormThreads;
        v[i] = k < d4 ? x[k] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kNormVec; i++) {
        ss += v[i].x * v[i].x;
        ss += v[i].y * v[i].y;
        ss += v[i].z * v[i].z;
        ss += v[i].w * v[i].w;
    }
    ss = warp_sum(ss);
    __shared__ float part[kNormThreads / 32];
    __shared__ float s_r;
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kNormThreads / 32; i++) t += part[i];
        s_r = rsqrtf(t / (float)d + eps);
    }
    __syncthreads();
    const float rr = s_r;
#pragma unroll
    for (int i = 0; i < kNormVec; i++) {
        const int k = threadIdx.x + i * kNormThreads;
        if (k < d4) {
            const int e = 4 * k;
            store4(out + (size_t)r * d + e, v[i].x * rr * to_f(w[e]), v[i].y * rr * to_f(w[e + 1]),
                   v[i].z * rr * to_f(w[e + 2]), v[i].w * rr * to_f(w[e + 3]));
        }
    }
}

template <typename T>
void launch_rmsnorm(cudaStream_t s, const float* X, const T* w, T* out, int rows, int d, float eps)
{
    launch_pdl(k_rmsnorm<T>, dim3(rows), dim3(kNormThreads), 0, s, X, w, out, d, eps);
}

// ---------------------------------------------------------- SIMT GEMMs ---
// out[r][o] = sum_k A[r][k] * W[o][k].  One warp per output feature o; lane
// partial sums over k = lane, lane+32, ... ascending, then a fixed xor tree.
// Rows are processed in register blocks of 8; the per-(r,o) order does not
// depend on the number of rows.
constexpr int kRB = 8;

template <typename T, int MODE>
__global__ void k_gemm_simt(const T* A, const T* W, const T* W2, float* outf, T* outt, int ld_out, int rows, int K,
                            int Nout)
{
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int o = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; o < Nout; o += warps) {
        const T* w = W + (size_t)o * K;
        const T* w2 = (MODE == 2) ? W2 + (size_t)o * K : nullptr;
        for (int r0 = 0; r0 < rows; r0 += kRB) {
            float acc[kRB], acc2[kRB];
#pragma unroll
            for (int i = 0; i < kRB; i++) acc[i] = acc2[i] = 0.f;
            for (int k = lane; k < K; k += 32) {
                float wk = to_f(w[k]);
                float wk2 = (MODE == 2) ? to_f(w2[k]) : 0.f;
#pragma unroll
                for (int i = 0; i < kRB; i++) {
                    if (r0 + i < rows) {
                        float a = to_f(A[(size_t)(r0 + i) * K + k]);
                        acc[i] += a * wk;
                        if (MODE == 2) acc2[i] += a * wk2;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kRB; i++) {
                float v = warp_sum(acc[i]);
                float v2 = (MODE == 2) ? warp_sum(acc2[i]) : 0.f;
                if (lane == 0 && r0 + i < rows) {
                    size_t idx = (size_t)(r0 + i) * ld_out + o;
                    if (MODE == 0) outf[idx] = v;
                    else if (MODE == 1) outf[idx] = outf[idx] + v;
                    else outt[idx] = from_f<T>(v / (1.0f + expf(-v)) * v2);
                }
            }
        }
    }
}

static int simt_blocks(int Nout) { return ceil_div(Nout, 8) < 4096 ? ceil_div(Nout, 8) : 4096; }

template <typename T>
void launch_gemm_simt_f32out(cudaStream_t s, const T* A, const T* W, float* out, int ld_out, int rows, int K,
                             int Nout)
{
    k_gemm_simt<T, 0><<<simt_blocks(Nout), 256, 0, s>>>(A, W, nullptr, out, nullptr, ld_out, rows, K, Nout);
}

template <typename T>
void launch_gemm_simt_resid(cudaStream_t s, const T* A, const T* W, float* X, int rows, int K, int Nout)
{
    k_gemm_simt<T, 1><<<simt_blocks(Nout), 256, 0, s>>>(A, W, nullptr, X, nullptr, Nout, rows, K, Nout);
}

template <typename T>
void launch_gemm_simt_swiglu(cudaStream_t s, const T* A, const T* Wg, const T* Wu, T* out, int rows, int K, int F)
{
    k_gemm_simt<T, 2><<<simt_blocks(F), 256, 0, s>>>(A, Wg, Wu, nullptr, out, F, rows, K, F);
}

// ----------------------------------------------------------------- RoPE ---
// qkv: fp32 [rows][H*hd + 2*Hkv*hd] straight from the projections.
// Rotate-half pairs (i, i + hd/2) of every q and k head at the row's
// position; write Q [rows][H][hd], K/V [rows][Hkv][hd] in T.
template <typename T>
__global__ void k_rope_split(const float* qkv, const int* pos, const float* cosb, const float* sinb, T* Q, T* KS,
                             T* VS, int H, int Hkv, int hd)
{
    const int r = blockIdx.x, half = hd / 2;
    const int dq = H * hd, dkv = Hkv * hd, ld = dq + 2 * dkv;
    const float* x = qkv + (size_t)r * ld;
    const int p = pos[r];
    for (int e = threadIdx.x; e < (H + Hkv) * half; e += blockDim.x) {
        int h = e / half, i = e - h * half;
        float c = cosb[(size_t)p * half + i], sn = sinb[(size_t)p * half + i];
        const float* v = x + h * hd;  // heads of q, then heads of k (contiguous)
        float x1 = v[i], x2 = v[i + half];
        float y1 = x1 * c - x2 * sn, y2 = x2 * c + x1 * sn;
        if (h < H) {
            Q[(size_t)r * dq + h * hd + i] = from_f<T>(y1);
            Q[(size_t)r * dq + h * hd + i + half] = from_f<T>(y2);
        } else {
            int hk = h - H;
            KS[(size_t)r * dkv + hk * hd + i] = from_f<T>(y1);
            KS[(size_t)r * dkv + hk * hd + i + half] = from_f<T>(y2);
        }
    }
    for (int e = threadIdx.x; e < dkv; e += blockDim.x) VS[(size_t)r * dkv + e] = from_f<T>(x[dq + dkv + e]);
}

template <typename T>
void launch_rope_split(cudaStream_t s, const float* qkv, const int* pos, const float* cosb, const float* sinb, T* Q,
                       T* KS, T* VS, int rows, int H, int Hkv, int hd)
{
    k_rope_split<T><<<rows, 128, 0, s>>>(qkv, pos, cosb, sinb, Q, KS, VS, H, Hkv, hd);
}

// ------------------------------------------------------------ attention ---
// One warp per (row, head).  Row r (group grp[r], position P + rel_pos[r])
// sees the cache [0,P) and, at position P + o for o <= rel_pos[r], the key of
// step row grp_map[grp[r]][o].  Keys are walked in chunks of 32 absolute
// positions, one key per lane, with an online softmax (running max, rescale
// by exp(m_old - m_new)).
template <typename T>
__global__ void k_attn_simt(const DState* st, RowSet rs, const int* pos, const T* Q, const T* KC, const T* VC,
                            const T* KS, const T* VS, T* out, int H, int Hkv, int hd, int max_seq, float scale)
{
    const int r = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
    const int kvh = h / (H / Hkv), dq = H * hd, dkv = Hkv * hd;
    const int P = st->P, my_pos = pos[r], rel = rs.rel_pos[r];
    const int* gmap = rs.grp_map + (size_t)rs.grp[r] * rs.maxoff;
    __shared__ float qs[128];
    for (int e = lane; e < hd; e += 32) qs[e] = to_f(Q[(size_t)r * dq + h * hd + e]);
    __syncwarp();
    const T* kc = KC + (size_t)kvh * max_seq * hd;
    const T* vc = VC + (size_t)kvh * max_seq * hd;
    float m = -INFINITY, l = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int nd = hd / 32;
    for (int c0 = 0; c0 <= my_pos; c0 += 32) {
        const int p = c0 + lane;
        const T* krow = nullptr;
        const T* vrow = nullptr;
        if (p < P) {
            krow = kc + (size_t)p * hd;
            vrow = vc + (size_t)p * hd;
        } else if (p - P <= rel) {
            int srow = gmap[p - P];
            krow = KS + (size_t)srow * dkv + kvh * hd;
            vrow = VS + (size_t)srow * dkv + kvh * hd;
        }
        float sc = -INFINITY;
        if (krow) {
            float a = 0.f;
            for (int e = 0; e < hd; e++) a += qs[e] * to_f(krow[e]);
            sc = a * scale;
        }
        const float m_new = fmaxf(m, warp_max(sc));
        const float alpha = expf(m - m_new);
        const float pr = krow ? expf(sc - m_new) : 0.f;
        l = l * alpha + warp_sum(pr);
        for (int i = 0; i < nd; i++) acc[i] *= alpha;
        const unsigned vis = __ballot_sync(0xffffffffu, krow != nullptr);
        for (int k = 0; k < 32; k++) {
            const float pk = __shfl_sync(0xffffffffu, pr, k);
            const T* vk = (const T*)__shfl_sync(0xffffffffu, (unsigned long long)vrow, k);
            if (vis & (1u << k))
                for (int i = 0; i < nd; i++) acc[i] += pk * to_f(vk[lane + 32 * i]);
        }
        m = m_new;
    }
    for (int i = 0; i < nd; i++) out[(size_t)r * dq + h * hd + lane + 32 * i] = from_f<T>(acc[i] / l);
}

template <typename T>
void launch_attn_simt(cudaStream_t s, const DState* st, RowSet rs, const int* pos, const T* Q, const T* KC,
                      const T* VC, const T* KS, const T* VS, T* out, int rows, int H, int Hkv, int hd, int max_seq,
                      float scale)
{
    dim3 grid(rows, H);
    k_attn_simt<T><<<grid, 32, 0, s>>>(st, rs, pos, Q, KC, VC, KS, VS, out, H, Hkv, hd, max_seq, scale);
}

// --------------------------------------------------------------- argmax ---
// Lowest index of the maximum (order-independent comparison).
__global__ void k_argmax(const float* logits, int* amax, int V)
{
    const int r = blockIdx.x;
    const float* x = logits + (size_t)r * V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
        float t = x[v];
        if (t > bv || (t == bv && v < bi)) { bv = t; bi = v; }
    }
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    __shared__ float sv[32];
    __shared__ int si[32];
    if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = bv; si[threadIdx.x >> 5] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); w++)
            if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) { bv = sv[w]; bi = si[w]; }
        amax[r] = bi;
    }
}

void launch_argmax(cudaStream_t s, const float* logits, int* amax, int rows, int V)
{
    k_argmax<<<rows, 256, 0, s>>>(logits, amax, V);
}

// ------------------------------------------------------ instantiations ---
#define LA_INST(T)                                                                                              \
    template void launch_embed<T>(cudaStream_t, const int*, const T*, float*, int, int);                        \
    template void launch_rmsnorm<T>(cudaStream_t, const float*, const T*, T*, int, int, float);                 \
    template void launch_gemm_simt_f32out<T>(cudaStream_t, const T*, const T*, float*, int, int, int, int);     \
    template void launch_gemm_simt_resid<T>(cudaStream_t, const T*, const T*, float*, int, int, int);           \
    template void launch_gemm_simt_swiglu<T>(cudaStream_t, const T*, const T*, const T*, T*, int, int, int);    \
    template void launch_rope_split<T>(cudaStream_t, const float*, const int*, const float*, const float*, T*,  \
                                       T*, T*, int, int, int, int);                                             \
    template void launch_attn_simt<T>(cudaStream_t, const DState*, RowSet, const int*, const T*, const T*,      \
                                      const T*, const T*, const T*, T*, int, int, int, int, int, float);
LA_INST(float)
LA_INST(__nv_bfloat16)

}  // namespace la
