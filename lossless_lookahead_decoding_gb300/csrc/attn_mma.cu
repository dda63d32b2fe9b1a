// attn_mma.cu -- masked lookahead / verification attention on tensor cores.
//
// The combined step's rows attend to the KV cache [0,P) (shared by every
// row) and to a few in-step rows: row r of group g sees, at position P + o
// (o <= rel_pos[r]), the step row grp_map[g][o] (the 2D-window + verification
// mask of the lookahead step; a prefill block is one causal group).
//
// Keys are walked in chunks of 64 ABSOLUTE positions; chunks are grouped into
// fixed splits of 256 positions (one CTA each) whose partial softmax states (max, sum,
// unnormalised output) are merged in ascending split order by a second
// kernel.  Inside a chunk, S = Q K^T and O += P V run on bf16 mma.sync tiles
// with fp32 accumulation.  A chunk that lies entirely below P is shared by
// all rows (16-row slabs, one per warp); a chunk that reaches P is a "tail"
// chunk: for every row group a warp builds the chunk's 64 key slots from the
// cache (positions < P) and from that group's step rows (positions >= P) by
// per-lane ldmatrix row addresses, so that slot j always holds position
// c*64 + j.  Every row therefore sees exactly the arithmetic it would see if
// it were decoded alone by plain greedy decoding (chunk and split boundaries
// at the same absolute positions, same instruction shapes, same reduction
// order, exact fp32 state hand-off), which keeps lookahead output identical
// to greedy output.
//
// The split that holds the first tail chunk is run by kRep CTAs: each
// repeats the split's shared chunks and then takes a share of the row
// groups, so the per-group work is spread over more SMs.
//
// Batched decoding with at most 16 rows per sequence (greedy batches: one)
// runs a narrow instance instead: a 16-row tile, no replicas, 4 warps and
// 108 KB of shared memory (two CTAs per SM), or for at most 8 rows 2 warps,
// two chunk buffers, 8 step rows and 72 KB (three per SM).  There one warp computes per
// CTA, so the SM's number of resident CTAs sets how many (sequence, head,
// split) items progress at once; every row's arithmetic is the wide
// instance's (the same chunks, instructions and order).
#include <type_traits>

#include "common.cuh"

namespace la {

namespace {

constexpr int kChunk = 64;
#ifndef LA_ATTN_SPLIT
#define LA_ATTN_SPLIT 256
#endif
#ifndef LA_ATTN_REP
#define LA_ATTN_REP 2
#endif
constexpr int kSplit = LA_ATTN_SPLIT;
constexpr int kWarps = 8;
constexpr int kRep = LA_ATTN_REP;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

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

// Row-major tile of HD bf16 per row, 16-byte chunks XOR-swizzled by row & 7.
template <int HD>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk)
{
    return base + row * (HD * 2) + ((chunk ^ (row & 7)) << 4);
}

// Softmax state of the two rows (g, g+8) a thread holds in a 16-row slab.
template <int HD>
struct SlabState {
    float m[2], l[2];
    float o[HD / 8][4];
};

// Per-lane key-row addressing of one chunk: the rows this lane feeds to
// ldmatrix (4 for K: key n2*16 + (lane&7) + ((lane>>4)<<3); 4 for V: key
// kk*16 + (lane&7) + (((lane>>3)&1)<<3)), as unswizzled row base addresses
// plus the row index that sets the swizzle phase.
struct KeyRows {
    uint32_t kb[4], vb[4];
    int ksw[4], vsw[4];
};

__device__ __forceinline__ int key_k(int n2, int lane) { return n2 * 16 + (lane & 7) + ((lane >> 4) << 3); }
__device__ __forceinline__ int key_v(int kk, int lane) { return kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3); }

// One 64-key chunk for one 16-row slab; vis(half, j) says whether the
// thread's row (g or g+8) sees slot j.  The arithmetic is identical for
// shared and tail chunks.
template <int HD, bool MASKED, typename VISF>
__device__ __forceinline__ void chunk_update(const uint32_t (*qf)[4], SlabState<HD>& st, const KeyRows& kr, VISF vis,
                                             float sl2)
{
    const int lane = threadIdx.x & 31;
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; n++) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ks++) {
#pragma unroll
        for (int n2 = 0; n2 < 4; n2++) {
            uint32_t b[4];
            ldsm_x4(b, kr.kb[n2] + (((2 * ks + ((lane >> 3) & 1)) ^ (kr.ksw[n2] & 7)) << 4));
            mma16816(s[2 * n2], qf[ks], b[0], b[1]);
            mma16816(s[2 * n2 + 1], qf[ks], b[2], b[3]);
        }
    }
    const int t = lane & 3;
    float cm[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; n++) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float v = s[n][i] * sl2;
            if (MASKED && !vis(i >> 1, n * 8 + 2 * t + (i & 1))) v = -INFINITY;
            s[n][i] = v;
            cm[i >> 1] = fmaxf(cm[i >> 1], v);
        }
    }
    float alpha[2], mu[2], rs[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; h++) {
        cm[h] = fmaxf(cm[h], __shfl_xor_sync(0xffffffffu, cm[h], 1));
        cm[h] = fmaxf(cm[h], __shfl_xor_sync(0xffffffffu, cm[h], 2));
        const float mn = fmaxf(st.m[h], cm[h]);
        mu[h] = (mn == -INFINITY) ? 0.f : mn;
        alpha[h] = exp2f(st.m[h] - mu[h]);
        st.m[h] = mn;
    }
#pragma unroll
    for (int n = 0; n < 8; n++) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float p = exp2f(s[n][i] - mu[i >> 1]);
            s[n][i] = p;
            rs[i >> 1] += p;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; h++) {
        rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
        rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
        st.l[h] = st.l[h] * alpha[h] + rs[h];
    }
#pragma unroll
    for (int d = 0; d < HD / 8; d++) {
        st.o[d][0] *= alpha[0];
        st.o[d][1] *= alpha[0];
        st.o[d][2] *= alpha[1];
        st.o[d][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
        uint32_t a[4];
        a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int d2 = 0; d2 < HD / 16; d2++) {
            uint32_t b[4];
            ldsm_x4_t(b, kr.vb[kk] + (((2 * d2 + (lane >> 4)) ^ (kr.vsw[kk] & 7)) << 4));
            mma16816(st.o[2 * d2], a, b[0], b[1]);
            mma16816(st.o[2 * d2 + 1], a, b[2], b[3]);
        }
    }
}

struct AttnArgs {
    const DState* st;
    RowSet rs;
    const int* pos;
    const __nv_bfloat16 *Q, *KC, *VC, *KS, *VS;
    float* part;  // [H][nsplit][128][2 + HD]; batched: [B][H][nsplit][rows][2 + HD]
    __nv_bfloat16* out;
    int rows, H, Hkv, max_seq, nsplit, max_rel;
    size_t sb;  // batched: byte stride between the sequences' decode states and caches (grid z = sequence)
    int hpc;    // query heads per CTA (of one KV head): their rows stacked in the Q tile
    float sl2;  // log2(e) / sqrt(hd)
};

// Shared memory: the Q tile, kBufs chunk buffers (K then V of one chunk; up
// to kBufs chunk loads in flight), the step rows' K and V, and the state
// hand-off (o in buffers 1..2 once the cached chunks are done, m and l apart).
// R: rows of the tile (kRows, or 16 for the narrow instances); NB chunk
// buffers; RS step rows.
constexpr int kBufs = 3;
constexpr int kNarrowRows = 16, kNarrowWarps = 4, kNarrow8Warps = 2;

template <int HD, int R = kRows, int NB = kBufs, int RS = R>
struct AttnSmem {
    static constexpr int RB = HD * 2, PS = HD + 4;  // global partial state: o[HD], m, l, 2 pad
    static constexpr int kQ = 0;                                  // Q tile [R][HD]
    static constexpr int kBuf0 = kQ + R * RB;                     // chunk buffers
    static constexpr int kBufBytes = 2 * kChunk * RB;             // K [kChunk][HD] then V
    static constexpr int kDumpO = kBuf0 + kBufBytes;              // o [R][HD] fp32 (buffers 1..)
    static_assert(R * HD * 4 <= (NB - 1) * kBufBytes, "hand-off fits the chunk buffers after the first");
    static constexpr int kKS = kBuf0 + NB * kBufBytes;            // step K [RS][HD]
    static constexpr int kVS = kKS + RS * RB;                     // step V
    static constexpr int kML = kVS + RS * RB;                     // m, l [R][2] fp32
    static constexpr int kZero = kML + R * 8;                     // one zero row
    static constexpr int kInts = kZero + RB;                      // group bookkeeping
    static constexpr int kBytes = kInts + (2 * R + 2) * 4;
};

// kBatch: grid z is the sequence of a batched step (one sequence: z = 0 and
// none of the per-sequence offsets is computed).  R rows per tile, W warps,
// NR CTAs for the split with the first tail chunk, NB chunk buffers, RS step
// rows, MB CTAs per SM (the wide instance: kRows, kWarps, kRep, kBufs, kRows,
// 1).
template <int HD, bool kBatch, int R = kRows, int W = kWarps, int NR = kRep, int NB = kBufs, int RS = R, int MB = 1>
__global__ void __launch_bounds__(W * 32, MB) k_attn_mma(AttnArgs a)
{
    pdl_wait();
    pdl_trigger();
    using L = AttnSmem<HD, R, NB, RS>;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RB = HD * 2, NCH = HD / 8, PS = L::PS;
    const uint32_t sb = su32(smem);
    float* dump_o = (float*)(smem + L::kDumpO);
    float* dump_ml = (float*)(smem + L::kML);
    int* gcnt = (int*)(smem + L::kInts);  // [R + 1] rows of each group (< a.rows)
    int* gslab = gcnt + R + 1;            // [R + 1] slab prefix over groups

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int dq = a.H * HD, dkv = a.Hkv * HD;
    // sequence b of a batch: its own decode state and cache, rows b*rows ..
    const int b = kBatch ? blockIdx.z : 0;
    const size_t row0 = (size_t)b * a.rows;
    const int P = seq_ptr(a.st, a.sb, b)->P, maxpos = P + a.max_rel;
    // blockIdx.y < nsplit: split y; beyond: extra CTAs for the split that
    // holds the first tail chunk (the chunk containing position P)
    // this CTA's query heads h0 .. h0 + hpc - 1 share KV head kvh; their rows
    // are stacked as virtual rows v = (h - h0) * rows + r (v < vrows <= 128):
    // the cached chunks serve every virtual row at once, since all read the
    // same keys; the arithmetic of each row is unchanged
    const int h0 = blockIdx.x * a.hpc, kvh = h0 / (a.H / a.Hkv), vrows = a.hpc * a.rows;
    const int tail_split = (P / kChunk) * kChunk / kSplit;
    const int sp = blockIdx.y < a.nsplit ? blockIdx.y : tail_split;
    const int rep = blockIdx.y < a.nsplit ? 0 : blockIdx.y - a.nsplit + 1;
    const int n_rep = sp == tail_split ? NR : 1;
    const int p0 = sp * kSplit;
    if (p0 > maxpos) return;
    const int c_begin = p0 / kChunk;
    const int c_end = min(p0 + kSplit, maxpos + kChunk) / kChunk;  // exclusive
    const int c_shared_end = min(c_end, max(c_begin, P / kChunk));
    const bool has_tail = c_shared_end < c_end;
    if (!has_tail && rep > 0) return;  // replicas only serve splits with tail chunks
    const __nv_bfloat16* kc = seq_ptr(a.KC, a.sb, b) + (size_t)kvh * a.max_seq * HD;
    const __nv_bfloat16* vc = seq_ptr(a.VC, a.sb, b) + (size_t)kvh * a.max_seq * HD;
    const __nv_bfloat16* qrows = a.Q + row0 * dq;
    const int* pos = a.pos + row0;
    // partials [B][H][nsplit][prow][PS]: one sequence keeps the 128-row stride
    const int prow = kBatch ? a.rows : kRows;
    float* part = a.part + row0 * a.H * a.nsplit * PS;
    // partial state of (virtual row v) in this split
    auto part_row = [&](int v) {
        const int hl = v / a.rows, r = v - hl * a.rows;
        return part + (((size_t)(h0 + hl) * a.nsplit + sp) * prow + r) * PS;
    };

    // Q tile: virtual rows of the CTA's heads (beyond vrows zero)
    for (int i = tid; i < R * NCH; i += blockDim.x) {
        const int v = i / NCH, c = i % NCH;
        const bool ok = v < vrows;
        const int hl = ok ? v / a.rows : 0, r = ok ? v - hl * a.rows : 0;
        cp_async16(swz<HD>(sb + L::kQ, v, c), qrows + (size_t)r * dq + (h0 + hl) * HD + c * 8, ok);
    }
    auto load_chunk = [&](int cidx, int kofs, int vofs, int valid_end) {
        for (int i = tid; i < kChunk * NCH; i += blockDim.x) {
            const int r = i / NCH, c = i % NCH, p = cidx * kChunk + r;
            const bool ok = p < valid_end;
            const size_t off = (size_t)(ok ? p : 0) * HD + c * 8;
            cp_async16(swz<HD>(sb + kofs, r, c), kc + off, ok);
            cp_async16(swz<HD>(sb + vofs, r, c), vc + off, ok);
        }
    };
    auto buf = [&](int i) { return L::kBuf0 + (i % NB) * L::kBufBytes; };
    // group 0: Q, and the step rows' K/V of this KV head when the CTA has tail work
    if (has_tail) {
        for (int i = tid; i < RS * NCH; i += blockDim.x) {
            const int r = i / NCH, c = i % NCH;
            const bool ok = r < a.rows;
            const size_t off = (row0 + (ok ? r : 0)) * dkv + kvh * HD + c * 8;
            cp_async16(swz<HD>(sb + L::kKS, r, c), a.KS + off, ok);
            cp_async16(swz<HD>(sb + L::kVS, r, c), a.VS + off, ok);
        }
    }
    cp_commit();
    // groups 1..NB: the first cached chunks (empty groups keep the count uniform)
    const int n_shared = c_shared_end - c_begin;
#pragma unroll
    for (int j = 0; j < NB; j++) {
        if (j < n_shared) load_chunk(c_begin + j, buf(j), buf(j) + kChunk * RB, P);
        cp_commit();
    }

    SlabState<HD> st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int d = 0; d < HD / 8; d++) st.o[d][0] = st.o[d][1] = st.o[d][2] = st.o[d][3] = 0.f;

    uint32_t qf[HD / 16][4];
    for (int i = 0; i < n_shared; i++) {
        cp_wait<NB - 1>();  // chunk i (and everything before it) has landed
        __syncthreads();
        if (warp * 16 < vrows) {  // slabs of padding rows only are skipped
            if (i == 0) {
#pragma unroll
                for (int ks = 0; ks < HD / 16; ks++)
                    ldsm_x4(qf[ks], swz<HD>(sb + L::kQ, warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                            2 * ks + (lane >> 4)));
            }
            const uint32_t kt = sb + buf(i), vt = kt + kChunk * RB;
            KeyRows kr;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                kr.kb[j] = kt + key_k(j, lane) * RB;
                kr.ksw[j] = key_k(j, lane);
                kr.vb[j] = vt + key_v(j, lane) * RB;
                kr.vsw[j] = key_v(j, lane);
            }
            chunk_update<HD, false>(qf, st, kr, [](int, int) { return true; }, a.sl2);
        }
        __syncthreads();  // buffer i is free again
        if (i + NB < n_shared) load_chunk(c_begin + i + NB, buf(i), buf(i) + kChunk * RB, P);
        cp_commit();
    }
    // state after the shared chunks: final partial, or hand-off to the tail
    if (has_tail) {
        cp_wait<0>();
        __syncthreads();  // chunk buffers 1, 2 become the hand-off
    }
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
            const int v = warp * 16 + g + 8 * hh;
            if (v < vrows) {
                float* po = has_tail ? dump_o + (size_t)v * HD : part_row(v);
                float* pml = has_tail ? dump_ml + 2 * v : part_row(v) + HD;
                if (t == 0) *(float2*)pml = make_float2(st.m[hh], st.l[hh]);
#pragma unroll
                for (int d = 0; d < HD / 8; d++)
                    *(float2*)(po + d * 8 + 2 * t) = make_float2(st.o[d][2 * hh], st.o[d][2 * hh + 1]);
            }
        }
    }
    if (!has_tail) return;

    // ---------------- tail chunks: per row group
    const int tile0 = c_shared_end * kChunk;  // first tail chunk's cache rows (buffer 0)
    load_chunk(c_shared_end, L::kBuf0, L::kBuf0 + kChunk * RB, P);
    cp_commit();
    if (tid < NCH) *(uint4*)(smem + L::kZero + tid * 16) = make_uint4(0, 0, 0, 0);
    // rows of each group, in row order (static lists, clipped to a.rows)
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
    cp_wait<0>();
    __syncthreads();
    const int n_group_items = gslab[ng], n_items = a.hpc * n_group_items;
    const int g4 = lane >> 2;
    for (int it_all = rep * W + warp; it_all < n_items; it_all += n_rep * W) {
        // item = (head of the CTA, slab of a row group); rows r, virtual rows hl * rows + r
        const int hl = it_all / n_group_items, it = it_all - hl * n_group_items, vofs = hl * a.rows;
        int g = 0;
        while (gslab[g + 1] <= it) g++;
        const int* glist = a.rs.grp_rows + a.rs.grp_start[g];
        const int r_begin = (it - gslab[g]) * 16, r_end = gcnt[g];
        // rows of this slab (-1 = padding)
        const int rA = (r_begin + g4 < r_end) ? glist[r_begin + g4] : -1;
        const int rB = (r_begin + g4 + 8 < r_end) ? glist[r_begin + g4 + 8] : -1;
        const int posA = rA >= 0 ? pos[rA] : -1, posB = rB >= 0 ? pos[rB] : -1;
        // Q fragments of the gathered rows
        {
            const int li = (lane & 7) + (((lane >> 3) & 1) << 3);
            const int rq = (r_begin + li < r_end) ? glist[r_begin + li] : -1;
#pragma unroll
            for (int ks = 0; ks < HD / 16; ks++) {
                const int ch = 2 * ks + (lane >> 4);
                ldsm_x4(qf[ks], rq >= 0 ? swz<HD>(sb + L::kQ, vofs + rq, ch) : sb + L::kZero + (ch << 4));
            }
        }
        // resume the rows' states (exact fp32 hand-off)
        SlabState<HD> ts;
        {
            const int t = lane & 3;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int r = hh ? rB : rA;
                if (r >= 0) {
                    const float* pr = dump_o + (size_t)(vofs + r) * HD;
                    ts.m[hh] = dump_ml[2 * (vofs + r)];
                    ts.l[hh] = dump_ml[2 * (vofs + r) + 1];
#pragma unroll
                    for (int d = 0; d < HD / 8; d++) {
                        const float2 v = *(const float2*)(pr + d * 8 + 2 * t);
                        ts.o[d][2 * hh] = v.x;
                        ts.o[d][2 * hh + 1] = v.y;
                    }
                } else {
                    ts.m[hh] = -INFINITY;
                    ts.l[hh] = 0.f;
#pragma unroll
                    for (int d = 0; d < HD / 8; d++) ts.o[d][2 * hh] = ts.o[d][2 * hh + 1] = 0.f;
                }
            }
        }
        const int* gmap = a.rs.grp_map + (size_t)g * a.rs.maxoff;
        for (int c = c_shared_end; c < c_end; c++) {
            const int c0 = c * kChunk;
            // slot j -> cache tile row, this group's step row, or the zero row
            KeyRows kr;
#pragma unroll
            for (int half = 0; half < 2; half++) {
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int key = half ? key_v(j, lane) : key_k(j, lane);
                    const int p = c0 + key;
                    int row = 0;
                    uint32_t kb, vb;
                    if (p < P) {
                        row = p - tile0;
                        kb = sb + L::kBuf0 + row * RB;
                        vb = sb + L::kBuf0 + kChunk * RB + row * RB;
                    } else if (p - P < a.rs.maxoff) {
                        row = gmap[p - P];
                        kb = sb + L::kKS + row * RB;
                        vb = sb + L::kVS + row * RB;
                    } else {
                        kb = vb = sb + L::kZero;
                    }
                    if (half) {
                        kr.vb[j] = vb;
                        kr.vsw[j] = row;
                    } else {
                        kr.kb[j] = kb;
                        kr.ksw[j] = row;
                    }
                }
            }
            chunk_update<HD, true>(qf, ts, kr, [&](int hh, int j) { return c0 + j <= (hh ? posB : posA); }, a.sl2);
        }
        {
            const int t = lane & 3;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int r = hh ? rB : rA;
                if (r >= 0) {
                    float* pr = part_row(vofs + r);
                    if (t == 0) *(float2*)(pr + HD) = make_float2(ts.m[hh], ts.l[hh]);
#pragma unroll
                    for (int d = 0; d < HD / 8; d++)
                        *(float2*)(pr + d * 8 + 2 * t) = make_float2(ts.o[d][2 * hh], ts.o[d][2 * hh + 1]);
                }
            }
        }
    }
}

// Merge the splits of every (row, head) in ascending split order.  One warp
// per (row, head), each lane HD/32 consecutive output dims; the loads of up
// to 4 splits are issued together, the merge runs in split order.
constexpr int kCombWarps = 8;

template <int HD, bool kBatch>
__global__ void __launch_bounds__(kCombWarps * 32, 5) k_attn_combine(AttnArgs a)
{
    pdl_wait();
    pdl_trigger();
    constexpr int PS = HD + 4, V = HD / 32, kB = 4;  // few registers: the whole grid fits in one wave
    using VecT = typename std::conditional<V == 4, float4, float2>::type;
    const int w = blockIdx.x * kCombWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= a.rows * a.H) return;
    const int r = w / a.H, h = w % a.H;
    const size_t row0 = kBatch ? (size_t)blockIdx.y * a.rows : 0;  // sequence blockIdx.y of a batch
    const int ns = a.pos[row0 + r] / kSplit + 1;
    const int prow = kBatch ? a.rows : kRows;  // the partials' row stride (k_attn_mma)
    const float* base = a.part + row0 * a.H * a.nsplit * PS + ((size_t)h * a.nsplit * prow + r) * PS;
    const size_t stride = (size_t)prow * PS;
    float m = -INFINITY, l = 0.f, o[V];
#pragma unroll
    for (int k = 0; k < V; k++) o[k] = 0.f;
    for (int s0 = 0; s0 < ns; s0 += kB) {
        float2 ml[kB];
        VecT ov[kB];
#pragma unroll
        for (int j = 0; j < kB; j++) {
            const bool ok = s0 + j < ns;
            const float* pr = base + (size_t)(ok ? s0 + j : 0) * stride;
            ml[j] = ok ? *(const float2*)(pr + HD) : make_float2(-INFINITY, 0.f);
            ov[j] = *(const VecT*)(pr + lane * V);
        }
#pragma unroll
        for (int j = 0; j < kB; j++) {
            if (s0 + j >= ns) break;
            const float* os = (const float*)&ov[j];
            if (s0 + j == 0) {
                m = ml[j].x;
                l = ml[j].y;
#pragma unroll
                for (int k = 0; k < V; k++) o[k] = os[k];
                continue;
            }
            const float mn = fmaxf(m, ml[j].x);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float fa = exp2f(m - mu), fb = exp2f(ml[j].x - mu);
            l = l * fa + ml[j].y * fb;
#pragma unroll
            for (int k = 0; k < V; k++) o[k] = o[k] * fa + os[k] * fb;
            m = mn;
        }
    }
    __nv_bfloat16* dst = a.out + (row0 + r) * a.H * HD + h * HD + lane * V;
#pragma unroll
    for (int k = 0; k < V; k += 2) *(__nv_bfloat162*)(dst + k) = __floats2bfloat162_rn(o[k] / l, o[k + 1] / l);
}

}  // namespace

size_t attn_mma_partial_bytes(int H, int hd, int max_seq)
{
    const int nsplit = (max_seq + kSplit - 1) / kSplit;
    return (size_t)H * nsplit * kRows * (hd + 4) * 4;
}

bool attn_mma_init(int hd)
{
    auto set = [](auto kern, int bytes) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
    };
    // the narrow instances also ask for the largest shared-memory carveout (two or three CTAs per SM)
    auto set_narrow = [&](auto kern, int bytes) {
        return set(kern, bytes) &&
               cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
    };
    auto all = [&](auto hdc) {
        constexpr int HD = decltype(hdc)::value;
        return set(k_attn_mma<HD, false>, AttnSmem<HD>::kBytes) && set(k_attn_mma<HD, true>, AttnSmem<HD>::kBytes) &&
               set_narrow(k_attn_mma<HD, true, kNarrowRows, kNarrowWarps, 1>, AttnSmem<HD, kNarrowRows>::kBytes) &&
               set_narrow(k_attn_mma<HD, true, kNarrowRows, kNarrow8Warps, 1, 2, 8, 3>,
                          AttnSmem<HD, kNarrowRows, 2, 8>::kBytes);
    };
    if (hd == 128) return all(std::integral_constant<int, 128>());
    if (hd == 64) return all(std::integral_constant<int, 64>());
    return false;
}

void launch_attn_mma(cudaStream_t s, const DState* st, RowSet rs, int max_rel, const int* pos, const void* Q,
                     const void* KC, const void* VC, const void* KS, const void* VS, void* out, float* part, int rows,
                     int H, int Hkv, int hd, int max_seq, int B, size_t sb)
{
    AttnArgs a;
    a.sb = sb;
    a.st = st;
    a.rs = rs;
    a.pos = pos;
    a.Q = (const __nv_bfloat16*)Q;
    a.KC = (const __nv_bfloat16*)KC;
    a.VC = (const __nv_bfloat16*)VC;
    a.KS = (const __nv_bfloat16*)KS;
    a.VS = (const __nv_bfloat16*)VS;
    a.part = part;
    a.out = (__nv_bfloat16*)out;
    a.rows = rows;
    a.H = H;
    a.Hkv = Hkv;
    a.max_seq = max_seq;
    a.nsplit = (max_seq + kSplit - 1) / kSplit;
    a.max_rel = max_rel;
    a.sl2 = 1.4426950408889634f / sqrtf((float)hd);
    // the narrow instances: batches of at most 16 rows, and 16 row groups, per sequence
    const bool narrow = B > 1 && rows <= kNarrowRows && rs.ngrp <= kNarrowRows;
    const int tile = narrow ? kNarrowRows : kRows;
    // query heads per CTA: the largest power of two dividing the GQA group
    // whose stacked rows still fit the tile (1 without GQA)
    const int group = H / Hkv;
    a.hpc = 1;
    while (group % (2 * a.hpc) == 0 && 2 * a.hpc * rows <= tile) a.hpc *= 2;
    // the 2-warp instance (three CTAs per SM) for at most 8 rows once the CTAs
    // of one split outnumber the SMs; below that each CTA's own latency
    // counts and 4 warps load a chunk faster
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool narrow8 = narrow && rows <= 8 && B * (H / a.hpc) > sms;
    dim3 grid(H / a.hpc, a.nsplit + (narrow ? 0 : kRep - 1), B);
    dim3 cgrid((rows * H + kCombWarps - 1) / kCombWarps, B);
    auto go = [&](auto mma, auto comb, int smem, int warps) {
        launch_pdl(mma, grid, dim3(warps * 32), smem, s, a);
        launch_pdl(comb, cgrid, dim3(kCombWarps * 32), 0, s, a);
    };
    auto pick = [&](auto hdc) {
        constexpr int HD = decltype(hdc)::value;
        if (narrow8)
            go(k_attn_mma<HD, true, kNarrowRows, kNarrow8Warps, 1, 2, 8, 3>, k_attn_combine<HD, true>,
               AttnSmem<HD, kNarrowRows, 2, 8>::kBytes, kNarrow8Warps);
        else if (narrow)
            go(k_attn_mma<HD, true, kNarrowRows, kNarrowWarps, 1>, k_attn_combine<HD, true>,
               AttnSmem<HD, kNarrowRows>::kBytes, kNarrowWarps);
        else if (B == 1)
            go(k_attn_mma<HD, false>, k_attn_combine<HD, false>, AttnSmem<HD>::kBytes, kWarps);
        else
            go(k_attn_mma<HD, true>, k_attn_combine<HD, true>, AttnSmem<HD>::kBytes, kWarps);
    };
    if (hd == 128) pick(std::integral_constant<int, 128>());
    else pick(std::integral_constant<int, 64>());
}

}  // namespace la
