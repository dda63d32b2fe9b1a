// engine.cu -- the C ABI of liblookahead.so (include/lookahead.h): context and
// workspace, prefill, the combined lookahead decode step, generation, stats
// and debug accessors.
//
// Method: Fu et al. 2024, "Break the Sequential Dependency of LLM Inference
// Using Lookahead Decoding", summary page, "Summary" (one forward pass holds
// the lookahead branch over a 2D window and the verification branch over pool
// candidates; the output equals greedy decoding) and "Key points" (knobs W, N,
// G).  A step is a fixed launch sequence on one stream: row assembly + pool
// lookup, embedding, per layer RMSNorm -> QKV+RoPE -> masked attention ->
// O-proj+residual -> RMSNorm -> gate/up+SwiGLU -> down+residual, final norm +
// LM head + argmax, verify + harvest + window shift, KV commit, and one
// device-to-host copy of the emitted tokens.  All decode state lives on the
// device, so the sequence is captured once into a CUDA graph and replayed.
// A batched context runs B independent sequences through the same launches:
// the forward pass over all B*T rows, the per-sequence kernels with the
// sequence as a grid dimension, one strided copy of the B decode states.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/lookahead.h"
#include "common.cuh"
#include "gemm_tc.cuh"

using namespace la;

namespace {

struct Layout {
    size_t off[32];
    size_t total;
    int n;
    size_t add(size_t bytes)
    {
        size_t o = total;
        off[n++] = o;
        total += (bytes + 1023) & ~(size_t)1023;
        return o;
    }
};

int next_pow2_log2(int x)
{
    int l = 0;
    while ((1 << l) < x) l++;
    return l;
}

}  // namespace

struct la_ctx {
    la_model_desc d;
    std::vector<const void*> lw;
    int W = 0, N = 2, G = 0, T = 1, flags = 0;
    // batched decoding: B sequences share each step's forward pass (rows
    // b*T .. b*T+T-1 are sequence b's); their state blocks are sb bytes apart
    // and the views below (KC, VC, prompt, win, pool, st, AOVR) are sequence 0's
    int B = 1;
    size_t sb = 0;
    int dseq = 0;  // the sequence the debug accessors read
    uint64_t seed = 0;
    float tau = 0.f;              // > 0: sampling verification at this temperature
    int top_k = 0;                // > 0: ... from the top_k tokens of each row only
    unsigned int top_p24 = 1u << 24;  // < 2^24: ... then from the leading tokens holding top_p of their weight
    unsigned long long* SSTAT = nullptr;  // per-row softmax max (float bits) / integer weight total for sampling
    int* AOVR = nullptr;                  // debug argmax override: [0] on, [1..T] the rows' argmaxes
    cudaStream_t s = nullptr;
    bool bf16 = false, use_tc = false, use_attn_mma = false, use_attn_tc = false;
    AttnTcPlan atc{};  // the step's attention on the tensor cores (tensor maps, launch shape)
    int atc_cta_y = 1;                          // its cache kernel's grid.y for the step being enqueued
    int graph_cta_y = 0;                        // ... as captured in (or last set on) the graph
    cudaGraph_t graph = nullptr;                // the captured step (kept to update node grids)
    std::vector<cudaGraphNode_t> atc_nodes;     // its cache-kernel launches
    float* attn_part = nullptr;
    int esz = 4, dq = 0, dkv = 0;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    bool own_ws = false;
    // workspace views
    char *KC = nullptr, *VC = nullptr, *KS = nullptr, *VS = nullptr;
    char *XN = nullptr, *Q = nullptr, *ATT = nullptr, *HID = nullptr;
    float *X = nullptr, *QKV32 = nullptr, *LOGITS = nullptr, *cosb = nullptr, *sinb = nullptr;
    int *AMAX = nullptr, *tok = nullptr, *pos = nullptr, *prompt = nullptr, *win = nullptr;
    int *dbg = nullptr;
    unsigned long long* AMAXP = nullptr;
    RowSet rs_step{}, rs_pre{};
    PoolView pool{};
    DState* st = nullptr;
    DState* h_st = nullptr;
    TcPlan tc{};
    Profiler prof;
    int kernels_per_step = 0;
    // host side (per sequence: prefilled, P)
    std::vector<char> prefilled_seq;
    std::vector<int> P_seq;
    bool prefilled = false, have_step = false;  // every sequence prefilled; a step ran since
    int P_host = 0;
    la_stats stats{};
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    cudaGraphExec_t gexec = nullptr;
    std::string err;
    // host-side fault injection (LA_FAULT, read at la_create)
    int fault_kind = 0;  // 0 none, 1 timeout, 2 capacity
    long long fault_step = 0;
};

// Fault injection for tests of the error paths, from the host only (no
// kernel is made to fail or wait): LA_FAULT=alloc | badarg | timeout@K |
// capacity@K.  alloc / badarg make la_create fail as if the workspace
// allocation failed / the arguments were refused; timeout@K writes
// LA_ERR_TIMEOUT into the device status word before the K-th step since the
// last prefill (as a bounded device-side wait that gave up would), so that
// step returns it; capacity@K makes the K-th step report a full KV cache.
// Each fires once per context.
enum { FAULT_NONE = 0, FAULT_TIMEOUT = 1, FAULT_CAPACITY = 2, FAULT_ALLOC = 3, FAULT_BADARG = 4 };

static int parse_fault(long long* step)
{
    const char* f = getenv("LA_FAULT");
    *step = 0;
    if (!f || !*f) return FAULT_NONE;
    if (!strcmp(f, "alloc")) return FAULT_ALLOC;
    if (!strcmp(f, "badarg")) return FAULT_BADARG;
    const char* at = strchr(f, '@');
    if (!at) return FAULT_NONE;
    *step = atoll(at + 1);
    if (*step < 1) return FAULT_NONE;
    if (!strncmp(f, "timeout@", 8)) return FAULT_TIMEOUT;
    if (!strncmp(f, "capacity@", 9)) return FAULT_CAPACITY;
    return FAULT_NONE;
}

#define LA_CK(call)                                                                                    \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess) {                                                                       \
            ctx->err = std::string(#call) + ": " + cudaGetErrorString(e_);                             \
            return LA_ERR_CUDA;                                                                        \
        }                                                                                              \
    } while (0)

static int fail(la_ctx* ctx, int code, const char* msg)
{
    if (ctx) ctx->err = msg;
    return code;
}

static int step_rows(int W, int N, int G) { return 1 + (W + G) * (N - 1); }

static const char* check_desc(const la_model_desc* d, int W, int N, int G, int B = 1)
{
    if (!d) return "desc is NULL";
    if (d->n_layers < 1 || d->d_model < 64 || d->d_model % 64 || d->d_model > 8192)
        return "d_model must be a multiple of 64 in [64, 8192]";
    if (d->head_dim != 64 && d->head_dim != 128) return "head_dim must be 64 or 128";
    if (d->n_heads < 1 || d->n_kv_heads < 1 || d->n_heads % d->n_kv_heads) return "n_heads % n_kv_heads != 0";
    if (d->ffn < 8 || d->ffn % 8) return "ffn must be a positive multiple of 8";
    if (d->vocab < 2 || d->max_seq < 2) return "bad vocab or max_seq";
    if (d->dtype != LA_FP32 && d->dtype != LA_BF16) return "dtype must be LA_FP32 or LA_BF16";
    if (!d->emb || !d->layer_w || !d->final_norm || !d->lm_head) return "missing weight pointer";
    if (W < 0 || G < 0 || N < 2 || N > kMaxN) return "need W >= 0, G >= 0, 2 <= N <= 8";
    if (step_rows(W, N, G) > kRows) return "1 + (W+G)(N-1) must be <= 128";
    if (B < 1 || B * step_rows(W, N, G) > kRows) return "batch * (1 + (W+G)(N-1)) must be <= 128";
    if ((N - 1) * W > 127) return "window too large";
    return nullptr;
}

// One sequence's decode state: its KV cache, prompt, lookahead window, n-gram
// pool, device decode state and argmax override.  A batched context holds B
// such blocks back to back, sb bytes apart (seq_ptr / seq_pool).
struct SeqLayout {
    size_t kc, vc, prompt, win, pk, ent, slot, st, aovr, bytes;
};

static SeqLayout seq_layout(const la_model_desc* d, int W, int N, int G, int lg)
{
    const int esz = d->dtype == LA_BF16 ? 2 : 4;
    const size_t L = d->n_layers, dkv = (size_t)d->n_kv_heads * d->head_dim, cap = (size_t)1 << lg;
    const int n1 = N - 1;
    SeqLayout q{};
    size_t o = 0;
    auto add = [&](size_t bytes) {
        const size_t at = o;
        o += (bytes + 1023) & ~(size_t)1023;
        return at;
    };
    q.kc = add(L * dkv * d->max_seq * esz);                   // K cache [L][Hkv][max_seq][hd]
    q.vc = add(L * dkv * d->max_seq * esz);                   // V cache
    q.prompt = add((size_t)d->max_seq * 4);                   // prompt tokens
    q.win = add((size_t)(n1 * (W > 0 ? W : 1)) * 4);          // window [N-1][W]
    q.pk = add(cap * 4 * 3);                                  // pool keys, counts, bulk-insert firsts
    q.ent = add(cap * (size_t)(G > 0 ? G : 1) * n1 * 4);      // pool entries
    q.slot = add((size_t)d->max_seq * 4);                     // pool bulk-insert slots
    q.st = add(sizeof(DState));                               // decode state
    q.aovr = add((kRows + 1) * 4);                            // argmax override: [0] on, [1..] rows
    q.bytes = o;
    return q;
}

enum LayoutItem {
    L_SEQ, L_KS, L_VS, L_X, L_XN, L_QKV32, L_Q, L_ATT, L_HID, L_LOGITS, L_COS, L_SIN, L_AMAX, L_TOK, L_POS,
    L_RS_STEP, L_MAP_STEP, L_RS_PRE, L_MAP_PRE, L_DEBUG, L_AMAXP, L_GL_STEP, L_GL_PRE, L_ATTN_PART, L_SSTAT,
    L_COUNT
};

static Layout make_layout(const la_model_desc* d, int W, int N, int G, int B, int* pool_log2, SeqLayout* sq)
{
    const int esz = d->dtype == LA_BF16 ? 2 : 4;
    const size_t L = d->n_layers, dq = (size_t)d->n_heads * d->head_dim, dkv = (size_t)d->n_kv_heads * d->head_dim;
    const int lg = next_pow2_log2(2 * d->vocab < 64 ? 64 : 2 * d->vocab);
    if (pool_log2) *pool_log2 = lg;
    const SeqLayout q = seq_layout(d, W, N, G, lg);
    if (sq) *sq = q;
    Layout ly{};
    ly.add(q.bytes * B);                                 // L_SEQ: the sequences' blocks
    ly.add(L * kRows * dkv * esz);                       // L_KS step K [L][kRows][dkv]
    ly.add(L * kRows * dkv * esz);                       // L_VS step V
    ly.add((size_t)kRows * d->d_model * 4);              // L_X residual stream
    ly.add((size_t)kRows * d->d_model * esz);            // L_XN normalised rows
    ly.add((size_t)kRows * (dq + 2 * dkv) * 4);          // L_QKV32
    ly.add((size_t)kRows * dq * esz);                    // L_Q
    ly.add((size_t)kRows * dq * esz);                    // L_ATT
    ly.add((size_t)kRows * d->ffn * esz);                // L_HID
    ly.add((size_t)kRows * d->vocab * 4);                // L_LOGITS
    ly.add((size_t)d->max_seq * (d->head_dim / 2) * 4);  // L_COS
    ly.add((size_t)d->max_seq * (d->head_dim / 2) * 4);  // L_SIN
    ly.add(kRows * 4);                                   // L_AMAX
    ly.add(kRows * 4);                                   // L_TOK
    ly.add(kRows * 4);                                   // L_POS
    ly.add(kRows * 4 * 2);                               // L_RS_STEP rel_pos + grp
    ly.add((size_t)kRows * kRows * 4);                   // L_MAP_STEP grp_map
    ly.add(kRows * 4 * 2);                               // L_RS_PRE
    ly.add(kRows * 4);                                   // L_MAP_PRE
    ly.add(4096);                                        // L_DEBUG scratch
    ly.add(kRows * 8);                                   // L_AMAXP packed argmax
    ly.add((2 * kRows + 1) * 4);                         // L_GL_STEP group lists
    ly.add((2 * kRows + 1) * 4);                         // L_GL_PRE
    const size_t pa = attn_mma_partial_bytes(d->n_heads, d->head_dim, d->max_seq);
    const size_t pt = attn_tc_partial_bytes(d->n_heads, d->head_dim, d->max_seq);
    ly.add(pa > pt ? pa : pt);                           // L_ATTN_PART split partials
    ly.add(kRows * 24);                                  // L_SSTAT sampling row statistics (max, S, K)
    return ly;
}

// Static row tables of the combined step (rows in the order: current token,
// lookahead rows (l, j) = 1 + l*W + j at offset 1 + j + l, verification rows
// (g, i) = 1 + W(N-1) + g(N-1) + i at offset 1 + i).  Row groups: window
// column j -> group j, candidate g -> group W + g, row 0 -> group 0.  map[grp]
// gives, for each position offset o from P, the step row whose key the
// group's rows see there (column j: the level-0 rows of columns 0..j, then
// levels 1.. of column j; candidate g: its own rows).  groups lists every
// group's rows in row order ([ngrp + 1] starts, then the rows).
// Diagonal levels (LA_MASK_DIAG): lookahead row (l, j) sits at offset 1 + j
// and sees only its own level, so level l is group l (candidates follow) and
// its map holds the level's rows at offsets 1..W.
struct StepTables {
    int T = 1, maxoff = 1, ngrp = 1;
    std::vector<int> rel, grp, map, groups;
};

static StepTables step_tables(int W, int N, int G, bool diag = false)
{
    StepTables tb;
    const int n1 = N - 1;
    const int lgrp = diag ? (W > 0 ? n1 : 0) : W;  // groups of the lookahead rows
    tb.T = step_rows(W, N, G);
    tb.rel.assign(kRows, 0);
    tb.grp.assign(kRows, 0);
    for (int l = 0; l < n1; l++)
        for (int j = 0; j < W; j++) {
            const int r = 1 + l * W + j;
            tb.rel[r] = diag ? 1 + j : 1 + j + l;
            tb.grp[r] = diag ? l : j;
        }
    for (int g = 0; g < G; g++)
        for (int i = 0; i < n1; i++) {
            const int r = 1 + W * n1 + g * n1 + i;
            tb.rel[r] = 1 + i;
            tb.grp[r] = lgrp + g;
        }
    for (int r = 0; r < tb.T; r++) tb.maxoff = tb.rel[r] + 1 > tb.maxoff ? tb.rel[r] + 1 : tb.maxoff;
    tb.ngrp = lgrp + G > 0 ? lgrp + G : 1;
    tb.map.assign((size_t)tb.ngrp * tb.maxoff, 0);
    if (diag) {
        for (int l = 0; l < lgrp; l++) {
            int* m = &tb.map[(size_t)l * tb.maxoff];
            for (int jj = 0; jj < W; jj++) m[1 + jj] = 1 + l * W + jj;  // level l, columns in order
        }
    } else {
        for (int j = 0; j < W; j++) {
            int* m = &tb.map[(size_t)j * tb.maxoff];
            for (int jj = 0; jj <= j; jj++) m[1 + jj] = 1 + jj;         // level 0, columns 0..j
            for (int l = 1; l < n1; l++) m[1 + j + l] = 1 + l * W + j;  // levels 1.. of column j
        }
    }
    for (int g = 0; g < G; g++) {
        int* m = &tb.map[(size_t)(lgrp + g) * tb.maxoff];
        for (int i = 0; i < n1; i++) m[1 + i] = 1 + W * n1 + g * n1 + i;
    }
    tb.groups.assign(2 * kRows + 1, 0);
    int k = 0;
    for (int g = 0; g < tb.ngrp; g++) {
        tb.groups[g] = k;
        for (int r = 0; r < tb.T; r++)
            if (tb.grp[r] == g) tb.groups[kRows + 1 + k++] = r;
    }
    tb.groups[tb.ngrp] = k;
    return tb;
}

extern "C" size_t la_workspace_bytes(const la_model_desc* desc, int W, int N, int G)
{
    return la_workspace_bytes_batch(desc, W, N, G, 1);
}

extern "C" size_t la_workspace_bytes_batch(const la_model_desc* desc, int W, int N, int G, int batch)
{
    if (check_desc(desc, W, N, G, batch)) return 0;
    return make_layout(desc, W, N, G, batch, nullptr, nullptr).total;
}

// One forward pass over `rows` rows: nseq sequences from seq0 on, rows / nseq
// consecutive rows each (a prefill block: one sequence; a step: all B).
template <typename T>
static void forward(la_ctx* c, int rows, const RowSet& rs, bool logits, int seq0, int nseq)
{
    const la_model_desc& d = c->d;
    const int L = d.n_layers, D = d.d_model, H = d.n_heads, Hkv = d.n_kv_heads, hd = d.head_dim, F = d.ffn;
    const int dq = c->dq, dkv = c->dkv;
    cudaStream_t s = c->s;
    T* XN = (T*)c->XN;
    T* Q = (T*)c->Q;
    T* ATT = (T*)c->ATT;
    T* HID = (T*)c->HID;
    const float scale = 1.0f / sqrtf((float)hd);
    launch_embed<T>(s, c->tok, (const T*)d.emb, c->X, rows, D);
    // tensor-core path: the down projection's residual add is folded into the
    // next RMSNorm (tc_resid_rmsnorm), so it stays pending across the loop
    TcResid pend{};
    bool pending = false;
    auto norm = [&](const T* w, T* out) {
        if (pending) tc_resid_rmsnorm(c->tc, s, pend, c->X, w, out, D, d.rms_eps);
        else launch_rmsnorm<T>(s, c->X, w, out, rows, D, d.rms_eps);
        pending = false;
    };
    for (int l = 0; l < L; l++) {
        const T* const* w = (const T* const*)&c->lw[(size_t)l * 9];
        T* KS = (T*)c->KS + (size_t)l * kRows * dkv;
        T* VS = (T*)c->VS + (size_t)l * kRows * dkv;
        const T* KC = seq_ptr((const T*)c->KC, c->sb, seq0) + (size_t)l * dkv * d.max_seq;
        const T* VC = seq_ptr((const T*)c->VC, c->sb, seq0) + (size_t)l * dkv * d.max_seq;
        const DState* st = seq_ptr(c->st, c->sb, seq0);
        const int rps = rows / nseq;  // rows of one sequence
        if (pending) {
            norm(w[0], XN);
        } else {
            c->prof.begin(s);
            launch_rmsnorm<T>(s, c->X, w[0], XN, rows, D, d.rms_eps);
            c->prof.end(s, P_NORM, 0, 0);
        }
        if (c->use_tc) {
            tc_qkv_rope(c->tc, s, l, rows, c->pos, c->cosb, c->sinb, (void*)Q, (void*)KS, (void*)VS);
        } else {
            const int ld = dq + 2 * dkv;
            launch_gemm_simt_f32out<T>(s, XN, w[1], c->QKV32, ld, rows, D, dq);
            launch_gemm_simt_f32out<T>(s, XN, w[2], c->QKV32 + dq, ld, rows, D, dkv);
            launch_gemm_simt_f32out<T>(s, XN, w[3], c->QKV32 + dq + dkv, ld, rows, D, dkv);
            launch_rope_split<T>(s, c->QKV32, c->pos, c->cosb, c->sinb, Q, KS, VS, rows, H, Hkv, hd);
        }
        c->prof.begin(s);
        if (c->use_attn_tc && &rs == &c->rs_step)
            launch_attn_tc(s, c->atc, l, l * kRows, c->st, rs, rs.maxoff - 1, c->pos, (const void*)Q, (void*)ATT,
                           c->attn_part, rows, &c->st->status, c->atc_cta_y);
        else if (c->use_attn_mma)
            launch_attn_mma(s, st, rs, &rs == &c->rs_pre ? rows - 1 : rs.maxoff - 1, c->pos, (const void*)Q,
                            (const void*)KC, (const void*)VC, (const void*)KS, (const void*)VS, (void*)ATT,
                            c->attn_part, rps, H, Hkv, hd, d.max_seq, nseq, c->sb);
        else
            for (int k = 0; k < nseq; k++) {
                const size_t r0 = (size_t)k * rps;
                launch_attn_simt<T>(s, seq_ptr(st, c->sb, k), rs, c->pos + r0, Q + r0 * dq, seq_ptr(KC, c->sb, k),
                                    seq_ptr(VC, c->sb, k), KS + r0 * dkv, VS + r0 * dkv, ATT + r0 * dq, rps, H, Hkv,
                                    hd, d.max_seq, scale);
            }
        c->prof.end(s, P_ATTN, rows, 0);  // bytes filled in per step (they depend on P)
        if (c->use_tc) {
            pend = tc_oproj(c->tc, s, l, rows);
            pending = true;
            norm(w[5], XN);
        } else {
            launch_gemm_simt_resid<T>(s, ATT, w[4], c->X, rows, dq, D);
            c->prof.begin(s);
            launch_rmsnorm<T>(s, c->X, w[5], XN, rows, D, d.rms_eps);
            c->prof.end(s, P_NORM, 0, 0);
        }
        if (c->use_tc) {
            tc_gateup_swiglu(c->tc, s, l, rows);
            pend = tc_down(c->tc, s, l, rows);
            pending = true;
        } else {
            launch_gemm_simt_swiglu<T>(s, XN, w[6], w[7], HID, rows, D, F);
            launch_gemm_simt_resid<T>(s, HID, w[8], c->X, rows, F, D);
        }
    }
    if (logits) {
        if (pending) {
            norm((const T*)d.final_norm, XN);
        } else {
            c->prof.begin(s);
            launch_rmsnorm<T>(s, c->X, (const T*)d.final_norm, XN, rows, D, d.rms_eps);
            c->prof.end(s, P_NORM, 0, 0);
        }
        if (c->use_tc) {
            tc_lmhead_argmax(c->tc, s, rows, ((c->flags & LA_DEBUG_LOGITS) || c->tau > 0.f) ? c->LOGITS : nullptr,
                             c->AMAXP, c->AMAX);
        } else {
            launch_gemm_simt_f32out<T>(s, XN, (const T*)d.lm_head, c->LOGITS, d.vocab, rows, D, d.vocab);
            launch_argmax(s, c->LOGITS, c->AMAX, rows, d.vocab);
        }
    }
}

static void run_forward(la_ctx* c, int rows, const RowSet& rs, bool logits, int seq0, int nseq)
{
    if (c->bf16) forward<__nv_bfloat16>(c, rows, rs, logits, seq0, nseq);
    else forward<float>(c, rows, rs, logits, seq0, nseq);
}

// The step's launch sequence (no host synchronisation inside).
static void enqueue_step(la_ctx* c)
{
    c->prof.idx = 0;
    c->prof.begin(c->s);
    launch_build_rows(c->s, c->st, c->win, c->pool, c->W, c->N, c->G, c->T, c->rs_step.rel_pos, c->tok, c->pos,
                      c->B, c->sb);
    c->prof.end(c->s, P_CONTROL, 0, 0);
    run_forward(c, c->B * c->T, c->rs_step, true, 0, c->B);
    c->prof.begin(c->s);
    const int vbase = 1 + c->W * (c->N - 1);
    if (c->tau > 0.f) launch_row_stats(c->s, c->LOGITS, c->d.vocab, c->tau, vbase, c->T, c->SSTAT, c->B, c->top_k,
                                       c->top_p24);
    launch_verify_update(c->s, c->st, c->tok, c->AMAX, c->win, c->pool, c->W, c->N, c->G, c->LOGITS, c->d.vocab,
                         c->tau, c->SSTAT, (c->flags & LA_MASK_DIAG) != 0, c->AOVR, c->B, c->sb);
    launch_commit(c->s, c->st, false, 0, c->N, c->KS, c->VS, c->KC, c->VC, c->d.n_layers, c->d.n_kv_heads,
                  c->d.head_dim, c->d.max_seq, c->esz, c->B, c->T, c->sb);
    c->prof.end(c->s, P_CONTROL, 0, 0);
    if (c->B == 1)
        cudaMemcpyAsync(c->h_st, c->st, sizeof(DState), cudaMemcpyDeviceToHost, c->s);
    else  // one strided copy gathers the B decode states
        cudaMemcpy2DAsync(c->h_st, sizeof(DState), c->st, c->sb, sizeof(DState), c->B, cudaMemcpyDeviceToHost, c->s);
}

// Accumulate the last step's event timings (P_before = the step's cache
// lengths summed over the sequences).
static void collect_profile(la_ctx* c, double P_before)
{
    Profiler& pr = c->prof;
    const double esz = c->esz, dq = c->dq, dkv = c->dkv, T = c->T, B = c->B;
    for (size_t i = 0; i < pr.idx; i++) {
        ProfPoint& p = pr.pts[i];
        float ms = 0.f;
        cudaEventElapsedTime(&ms, p.a, p.b);
        double by = p.bytes, fl = p.flops;
        if (p.cls == P_ATTN) {
            // the cache [0,P) once per KV head, plus the rows' q, k, v and output
            by = (2.0 * P_before * dkv + B * T * (2 * dq + 2 * dkv)) * esz;
            fl = 4.0 * T * (P_before + B) * dq;
        }
        pr.ms[p.cls] += ms;
        pr.bytes[p.cls] += by;
        pr.flops[p.cls] += fl;
        pr.n[p.cls] += 1;
    }
}

// The kernel nodes of a captured graph that launch `fn`.
static void find_kernel_nodes(cudaGraph_t g, const void* fn, std::vector<cudaGraphNode_t>* out)
{
    size_t n = 0;
    if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess || n == 0) return;
    std::vector<cudaGraphNode_t> nodes(n);
    if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return;
    for (size_t i = 0; i < n; i++) {
        cudaGraphNodeType t;
        cudaKernelNodeParams kp;
        if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel &&
            cudaGraphKernelNodeGetParams(nodes[i], &kp) == cudaSuccess && kp.func == fn)
            out->push_back(nodes[i]);
    }
}

// Count the kernel nodes of one captured step (the launches a step makes).
static int count_kernels(cudaGraph_t g)
{
    size_t n = 0;
    if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess || n == 0) return 0;
    std::vector<cudaGraphNode_t> nodes(n);
    if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return 0;
    int k = 0;
    for (size_t i = 0; i < n; i++) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) k++;
    }
    return k;
}

extern "C" int la_create(const la_model_desc* desc, int W, int N, int G, void* workspace, size_t ws_bytes,
                         uint64_t seed, int flags, la_ctx** out)
{
    return la_create_batch(desc, W, N, G, 1, workspace, ws_bytes, seed, flags, out);
}

extern "C" int la_create_batch(const la_model_desc* desc, int W, int N, int G, int batch, void* workspace,
                               size_t ws_bytes, uint64_t seed, int flags, la_ctx** out)
{
    if (!out) return LA_ERR_ARG;
    *out = nullptr;
    if (const char* why = check_desc(desc, W, N, G, batch)) {
        fprintf(stderr, "la_create: %s\n", why);
        return LA_ERR_ARG;
    }
    long long fault_step = 0;
    const int fault = parse_fault(&fault_step);
    if (fault == FAULT_BADARG) {
        fprintf(stderr, "la_create: arguments refused (injected by LA_FAULT)\n");
        return LA_ERR_ARG;
    }
    if (batch > 1 && (flags & LA_ATTN_TC)) {
        fprintf(stderr, "la_create: LA_ATTN_TC serves one sequence (batch 1)\n");
        return LA_ERR_ARG;
    }
    if (fault == FAULT_ALLOC) {
        fprintf(stderr, "la_create: workspace allocation failed (injected by LA_FAULT)\n");
        return LA_ERR_OOM;
    }
    la_ctx* ctx = new (std::nothrow) la_ctx();
    if (!ctx) return LA_ERR_OOM;
    ctx->fault_kind = fault;
    ctx->fault_step = fault_step;
    ctx->d = *desc;
    ctx->lw.assign(desc->layer_w, desc->layer_w + (size_t)desc->n_layers * 9);
    for (const void* p : ctx->lw)
        if (!p) {
            delete ctx;
            return LA_ERR_ARG;
        }
    ctx->d.layer_w = ctx->lw.data();
    ctx->W = W;
    ctx->N = N;
    ctx->G = G;
    ctx->T = step_rows(W, N, G);
    ctx->B = batch;
    ctx->prefilled_seq.assign(batch, 0);
    ctx->P_seq.assign(batch, 0);
    // the legacy default stream cannot be captured: launch directly there
    ctx->flags = desc->stream ? flags : (flags | LA_NO_GRAPH);
    ctx->seed = seed;
    ctx->s = (cudaStream_t)desc->stream;
    ctx->bf16 = desc->dtype == LA_BF16;
    ctx->esz = ctx->bf16 ? 2 : 4;
    ctx->dq = desc->n_heads * desc->head_dim;
    ctx->dkv = desc->n_kv_heads * desc->head_dim;
    int lg = 0;
    SeqLayout sq{};
    Layout ly = make_layout(desc, W, N, G, batch, &lg, &sq);
    ctx->sb = sq.bytes;
    if (workspace) {
        if (ws_bytes < ly.total || ((uintptr_t)workspace & 1023)) {
            delete ctx;
            return LA_ERR_ARG;
        }
        ctx->ws = (char*)workspace;
    } else {
        if (cudaMalloc((void**)&ctx->ws, ly.total) != cudaSuccess) {
            delete ctx;
            return LA_ERR_OOM;
        }
        ctx->own_ws = true;
    }
    ctx->ws_bytes = ly.total;
    char* b = ctx->ws;
    char* s0 = b + ly.off[L_SEQ];  // sequence 0's block
    ctx->KC = s0 + sq.kc;
    ctx->VC = s0 + sq.vc;
    ctx->prompt = (int*)(s0 + sq.prompt);
    ctx->win = (int*)(s0 + sq.win);
    int* pk = (int*)(s0 + sq.pk);
    const int cap = 1 << lg;
    ctx->st = (DState*)(s0 + sq.st);
    ctx->AOVR = (int*)(s0 + sq.aovr);
    ctx->pool = PoolView{pk, pk + cap, (int*)(s0 + sq.ent), pk + 2 * cap, (int*)(s0 + sq.slot),
                         &ctx->st->status, cap, lg, G, N - 1};
    ctx->KS = b + ly.off[L_KS];
    ctx->VS = b + ly.off[L_VS];
    ctx->X = (float*)(b + ly.off[L_X]);
    ctx->XN = b + ly.off[L_XN];
    ctx->QKV32 = (float*)(b + ly.off[L_QKV32]);
    ctx->Q = b + ly.off[L_Q];
    ctx->ATT = b + ly.off[L_ATT];
    ctx->HID = b + ly.off[L_HID];
    ctx->LOGITS = (float*)(b + ly.off[L_LOGITS]);
    ctx->cosb = (float*)(b + ly.off[L_COS]);
    ctx->sinb = (float*)(b + ly.off[L_SIN]);
    ctx->AMAX = (int*)(b + ly.off[L_AMAX]);
    ctx->tok = (int*)(b + ly.off[L_TOK]);
    ctx->pos = (int*)(b + ly.off[L_POS]);
    int* rs1 = (int*)(b + ly.off[L_RS_STEP]);
    int* map1 = (int*)(b + ly.off[L_MAP_STEP]);
    int* rs2 = (int*)(b + ly.off[L_RS_PRE]);
    int* map2 = (int*)(b + ly.off[L_MAP_PRE]);
    ctx->dbg = (int*)(b + ly.off[L_DEBUG]);
    ctx->AMAXP = (unsigned long long*)(b + ly.off[L_AMAXP]);
    int* gl1 = (int*)(b + ly.off[L_GL_STEP]);
    int* gl2 = (int*)(b + ly.off[L_GL_PRE]);
    ctx->attn_part = (float*)(b + ly.off[L_ATTN_PART]);
    ctx->SSTAT = (unsigned long long*)(b + ly.off[L_SSTAT]);

    // row tables: step (rows, positions and mask of the combined step) and prefill (causal)
    const StepTables tb = step_tables(W, N, G, (flags & LA_MASK_DIAG) != 0);
    const std::vector<int>&rel = tb.rel, &grp = tb.grp, &map = tb.map, &sgl = tb.groups;
    const int maxoff = tb.maxoff, ngrp = tb.ngrp;
    std::vector<int> prel(kRows), pgrp(kRows, 0), pmap(kRows);
    for (int r = 0; r < kRows; r++) prel[r] = pmap[r] = r;
    std::vector<int> pgl(2 * kRows + 1, 0);
    pgl[0] = 0;
    pgl[1] = kRows;
    for (int r = 0; r < kRows; r++) pgl[kRows + 1 + r] = r;
    std::vector<float> cs((size_t)desc->max_seq * (desc->head_dim / 2)), sn(cs.size());
    for (int p = 0; p < desc->max_seq; p++)
        for (int i = 0; i < desc->head_dim / 2; i++) {
            double ang = (double)p * std::pow((double)desc->rope_theta, -2.0 * i / (double)desc->head_dim);
            cs[(size_t)p * (desc->head_dim / 2) + i] = (float)std::cos(ang);
            sn[(size_t)p * (desc->head_dim / 2) + i] = (float)std::sin(ang);
        }
    int rc = LA_OK;
    {
        auto ck = [&](cudaError_t e) {
            if (e != cudaSuccess && rc == LA_OK) {
                ctx->err = cudaGetErrorString(e);
                rc = LA_ERR_CUDA;
            }
        };
        // zero the KV cache and the activations once: padded rows, and cache
        // positions not yet written that a tensor-core tile covers with zero
        // weight, must hold finite values
        // (with the sequences' blocks: decode states and argmax overrides start cleared)
        ck(cudaMemset(ctx->ws + ly.off[L_SEQ], 0, ly.off[L_COS] - ly.off[L_SEQ]));
        ck(cudaMemset(ctx->AMAXP, 0, kRows * 8));
        ck(cudaMemcpy(rs1, rel.data(), kRows * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(rs1 + kRows, grp.data(), kRows * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(map1, map.data(), map.size() * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(rs2, prel.data(), kRows * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(rs2 + kRows, pgrp.data(), kRows * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(map2, pmap.data(), kRows * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(gl1, sgl.data(), sgl.size() * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(gl2, pgl.data(), pgl.size() * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(ctx->cosb, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
        ck(cudaMemcpy(ctx->sinb, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
        ck(cudaHostAlloc((void**)&ctx->h_st, sizeof(DState) * batch, cudaHostAllocDefault));
        ck(cudaEventCreate(&ctx->ev0));
        ck(cudaEventCreate(&ctx->ev1));
    }
    ctx->rs_step = RowSet{rs1, rs1 + kRows, map1, gl1, gl1 + kRows + 1, maxoff, ngrp};
    ctx->rs_pre = RowSet{rs2, rs2 + kRows, map2, gl2, gl2 + kRows + 1, kRows, 1};
    if (rc == LA_OK && ctx->bf16 && !(flags & LA_SIMT)) {
        int trc = tc_plan_create(&ctx->tc, ctx->d, ctx->lw.data(), ctx->XN, ctx->Q, ctx->ATT, ctx->HID, ctx->esz,
                                 &ctx->st->status);
        ctx->tc.prof = &ctx->prof;
        if (trc == 0) {
            ctx->use_tc = true;
            ctx->use_attn_mma = attn_mma_init(desc->head_dim);
        }
        // the step's rows sit at most W + N - 2 positions past P (N - 1 for
        // candidate rows); the tensor-core attention keeps every row's recent
        // window of attn_tc_delta() positions out of its cache-only part
        if (trc == 0 && (flags & LA_ATTN_TC) && (W > 0 ? W + N - 2 : N - 1) > attn_tc_delta()) {
            ctx->err = "LA_ATTN_TC needs W + N - 2 <= 31";
            rc = LA_ERR_ARG;
        } else if (trc == 0 && (flags & LA_ATTN_TC)) {
            int items = 0;
            for (int g = 0; g < ngrp; g++) {
                int n = 0;
                for (int r = 0; r < tb.T; r++) n += grp[r] == g;
                items += (n + 15) / 16;
            }
            const long long kv_rows = (long long)desc->n_layers * desc->n_kv_heads * desc->max_seq;
            const int arc = !attn_tc_init(desc->head_dim)
                                ? LA_ERR_CUDA
                                : attn_tc_plan(&ctx->atc, ctx->Q, kRows, ctx->KC, ctx->VC, kv_rows, ctx->KS, ctx->VS,
                                               (long long)desc->n_layers * kRows, desc->n_heads, desc->n_kv_heads,
                                               desc->head_dim, desc->max_seq, tb.T, items);
            ctx->use_attn_tc = arc == LA_OK;
            // the pair prefers the largest shared-memory carveout; the GEMMs, their
            // epilogues and the residual norms then ask for it too, so that no SM
            // of the layer chain has to be reconfigured between kernels (with the
            // mma.sync attention the same setting was slower, so it is kept to
            // this path)
            if (ctx->use_attn_tc) ctx->tc.carveout = 100;
            if (arc == LA_ERR_ARG) {
                ctx->err = "max_seq must be <= 4096 on the bf16 tensor-core path";
                rc = LA_ERR_ARG;
            } else if (arc) {
                ctx->err = "tensor-core attention set-up failed";
                rc = LA_ERR_CUDA;
            }
        }
        else if (trc < 0) {
            ctx->err = "tcgen05 plan creation failed";
            rc = LA_ERR_CUDA;
        }
    }
    if (rc != LA_OK) {
        fprintf(stderr, "la_create: %s\n", ctx->err.c_str());
        la_destroy(ctx);
        return rc;
    }
    ctx->stats.rows = ctx->T * ctx->B;
    ctx->prof.on = (flags & LA_PROFILE) != 0;
    *out = ctx;
    return LA_OK;
}

extern "C" void la_destroy(la_ctx* ctx)
{
    if (!ctx) return;
    if (ctx->s) cudaStreamSynchronize(ctx->s);
    else cudaDeviceSynchronize();
    if (ctx->gexec) cudaGraphExecDestroy(ctx->gexec);
    if (ctx->graph) cudaGraphDestroy(ctx->graph);
    tc_plan_destroy(&ctx->tc);
    if (ctx->own_ws && ctx->ws) cudaFree(ctx->ws);
    if (ctx->h_st) cudaFreeHost(ctx->h_st);
    if (ctx->ev0) cudaEventDestroy(ctx->ev0);
    if (ctx->ev1) cudaEventDestroy(ctx->ev1);
    delete ctx;
}

extern "C" const char* la_last_error(la_ctx* ctx) { return ctx ? ctx->err.c_str() : "no context"; }

// splitmix64 (S. Vigna's published generator): the lookahead window is
// initialised from prompt tokens picked by this stream (level-major order).
static uint64_t splitmix64(uint64_t* x)
{
    uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Prefill of sequence `seq`: its prompt's KV into its cache, its window and
// pool initialised, its decode state reset.
static int prefill_seq(la_ctx* ctx, int seq, const int32_t* prompt, int len)
{
    if (!prompt || len < 1) return fail(ctx, LA_ERR_ARG, "prompt must hold at least one token");
    if (len + ctx->W + ctx->N > ctx->d.max_seq) return fail(ctx, LA_ERR_CAPACITY, "prompt too long for max_seq");
    for (int i = 0; i < len; i++)
        if (prompt[i] < 0 || prompt[i] >= ctx->d.vocab) return fail(ctx, LA_ERR_ARG, "token id out of range");
    ctx->prefilled = false;
    ctx->prefilled_seq[seq] = 0;
    cudaStream_t s = ctx->s;
    const size_t sb = ctx->sb;
    DState* st = seq_ptr(ctx->st, sb, seq);
    DState* h = ctx->h_st + seq;
    int* dprompt = seq_ptr(ctx->prompt, sb, seq);
    const PoolView pool = seq_pool(ctx->pool, sb, seq);
    LA_CK(cudaMemcpyAsync(dprompt, prompt, (size_t)len * 4, cudaMemcpyHostToDevice, s));
    std::vector<int> win((size_t)(ctx->N - 1) * (ctx->W > 0 ? ctx->W : 1), 0);
    uint64_t sm = ctx->seed;
    for (int l = 0; l < ctx->N - 1; l++)
        for (int j = 0; j < ctx->W; j++) win[(size_t)l * ctx->W + j] = prompt[splitmix64(&sm) % (uint64_t)len];
    LA_CK(cudaMemcpyAsync(seq_ptr(ctx->win, sb, seq), win.data(), win.size() * 4, cudaMemcpyHostToDevice, s));
    LA_CK(cudaStreamSynchronize(s));  // win is a host temporary
    launch_pool_reset(s, pool);
    launch_set_state(s, st, 0, prompt[len - 1], true);
    if ((ctx->flags & LA_PRESEED_PROMPT) && ctx->G > 0 && len >= ctx->N)
        launch_pool_insert(s, pool, dprompt, dprompt + 1, 1, len - ctx->N + 1);
    for (int P0 = 0; P0 < len - 1; P0 += kRows) {
        const int n = (len - 1 - P0) < kRows ? (len - 1 - P0) : kRows;
        launch_set_state(s, st, P0, prompt[len - 1], false);
        launch_prefill_rows(s, st, dprompt, P0, n, ctx->tok, ctx->pos);
        run_forward(ctx, n, ctx->rs_pre, false, seq, 1);
        launch_commit(s, st, true, n, n, ctx->KS, ctx->VS, seq_ptr(ctx->KC, sb, seq), seq_ptr(ctx->VC, sb, seq),
                      ctx->d.n_layers, ctx->d.n_kv_heads, ctx->d.head_dim, ctx->d.max_seq, ctx->esz);
    }
    launch_set_state(s, st, len - 1, prompt[len - 1], false);
    LA_CK(cudaGetLastError());
    LA_CK(cudaMemcpyAsync(h, st, sizeof(DState), cudaMemcpyDeviceToHost, s));
    LA_CK(cudaStreamSynchronize(s));
    if (h->status) return fail(ctx, h->status, "device status set during prefill");
    ctx->P_seq[seq] = len - 1;
    ctx->prefilled_seq[seq] = 1;
    bool all = true;
    for (char f : ctx->prefilled_seq) all = all && f;
    ctx->prefilled = all;
    ctx->have_step = false;
    if (seq == 0) memset(&ctx->stats, 0, sizeof(ctx->stats));  // sequence 0's prefill starts new statistics
    ctx->stats.prefill_tokens += len - 1;
    ctx->P_host = ctx->P_seq[0];
    ctx->stats.P = ctx->P_seq[0];
    ctx->stats.rows = ctx->T * ctx->B;
    return LA_OK;
}

extern "C" int la_prefill(la_ctx* ctx, const int32_t* prompt, int len)
{
    if (!ctx) return LA_ERR_ARG;
    if (ctx->B > 1) return fail(ctx, LA_ERR_STATE, "a batched context: use la_prefill_seq");
    return prefill_seq(ctx, 0, prompt, len);
}

extern "C" int la_prefill_seq(la_ctx* ctx, int seq, const int32_t* prompt, int len)
{
    if (!ctx) return LA_ERR_ARG;
    if (seq < 0 || seq >= ctx->B) return fail(ctx, LA_ERR_ARG, "seq out of range");
    return prefill_seq(ctx, seq, prompt, len);
}

// One combined step of every sequence: the step's graph (captured on first
// use), then the B decode states on the host.
static int run_step(la_ctx* ctx)
{
    if (!ctx->prefilled) return fail(ctx, LA_ERR_STATE, "la_step before every sequence was prefilled");
    for (int b = 0; b < ctx->B; b++)
        if (ctx->P_seq[b] + ctx->W + ctx->N > ctx->d.max_seq) return fail(ctx, LA_ERR_CAPACITY, "KV cache full");
    cudaStream_t s = ctx->s;
    // the attention's cache kernel: one CTA per split the step's rows reach
    if (ctx->use_attn_tc) ctx->atc_cta_y = attn_tc_splits(ctx->atc, ctx->P_host, ctx->rs_step.maxoff - 1);
    const int inject = (ctx->fault_kind && ctx->stats.steps + 1 == ctx->fault_step) ? ctx->fault_kind : 0;
    if (inject) ctx->fault_kind = FAULT_NONE;  // once per context
    if (inject == FAULT_CAPACITY) return fail(ctx, LA_ERR_CAPACITY, "KV cache full (injected)");
    if (inject == FAULT_TIMEOUT) {
        static const int code = LA_ERR_TIMEOUT;
        LA_CK(cudaMemcpyAsync(&ctx->st->status, &code, sizeof(int), cudaMemcpyHostToDevice, s));
    }
    LA_CK(cudaEventRecord(ctx->ev0, s));
    if (!(ctx->flags & LA_NO_GRAPH)) {
        if (!ctx->gexec) {
            cudaGraph_t g;
            LA_CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
            enqueue_step(ctx);
            cudaError_t e = cudaStreamEndCapture(s, &g);
            if (e != cudaSuccess) {
                ctx->err = std::string("graph capture: ") + cudaGetErrorString(e);
                return LA_ERR_CUDA;
            }
            ctx->kernels_per_step = count_kernels(g);
            e = cudaGraphInstantiate(&ctx->gexec, g, 0);
            if (e != cudaSuccess) {
                cudaGraphDestroy(g);
                ctx->gexec = nullptr;
                ctx->err = std::string("graph instantiate: ") + cudaGetErrorString(e);
                return LA_ERR_CUDA;
            }
            ctx->graph = g;
            ctx->atc_nodes.clear();
            if (ctx->use_attn_tc) find_kernel_nodes(g, attn_tc_cache_kernel(ctx->d.head_dim), &ctx->atc_nodes);
            ctx->graph_cta_y = ctx->atc_cta_y;
        }
        if (ctx->use_attn_tc && ctx->atc_cta_y != ctx->graph_cta_y) {
            // the split count changed with P: resize the cache kernel's grids
            for (cudaGraphNode_t node : ctx->atc_nodes) {
                cudaKernelNodeParams kp;
                LA_CK(cudaGraphKernelNodeGetParams(node, &kp));
                kp.gridDim.y = ctx->atc_cta_y;
                LA_CK(cudaGraphKernelNodeSetParams(node, &kp));
                LA_CK(cudaGraphExecKernelNodeSetParams(ctx->gexec, node, &kp));
            }
            ctx->graph_cta_y = ctx->atc_cta_y;
        }
        LA_CK(cudaGraphLaunch(ctx->gexec, s));
    } else {
        enqueue_step(ctx);
    }
    LA_CK(cudaEventRecord(ctx->ev1, s));
    LA_CK(cudaGetLastError());
    LA_CK(cudaEventSynchronize(ctx->ev1));
    for (int b = 0; b < ctx->B; b++) {
        const DState& h = ctx->h_st[b];
        if (h.status) {
            // the device state is not trusted after a device-side error: the
            // context needs la_prefill again (which clears the status word)
            ctx->prefilled = false;
            for (char& f : ctx->prefilled_seq) f = 0;
            return fail(ctx, h.status, "device status set during step");
        }
        if (h.n_emit < 1 || h.n_emit > ctx->N) return fail(ctx, LA_ERR_STATE, "corrupt step result");
    }
    double P_before = 0;
    for (int b = 0; b < ctx->B; b++) {
        const DState& h = ctx->h_st[b];
        ctx->P_seq[b] = h.P;
        ctx->stats.emitted += h.n_emit;
        ctx->stats.accept_hist[h.n_emit]++;
        P_before += h.P_before;
    }
    ctx->P_host = ctx->P_seq[0];
    ctx->have_step = true;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, ctx->ev0, ctx->ev1);
    ctx->stats.steps++;
    ctx->stats.P = ctx->P_seq[0];
    ctx->stats.last_step_ms = ms;
    ctx->stats.kernels_per_step = ctx->kernels_per_step;
    if (ctx->prof.on) collect_profile(ctx, P_before);
    return LA_OK;
}

extern "C" int la_step(la_ctx* ctx, int32_t* out, int cap, int* n_out)
{
    if (!ctx) return LA_ERR_ARG;
    if (ctx->B > 1) return fail(ctx, LA_ERR_STATE, "a batched context: use la_step_batch");
    if (!out || !n_out || cap < ctx->N) return fail(ctx, LA_ERR_ARG, "out must hold N tokens");
    const int rc = run_step(ctx);
    if (rc) return rc;
    const DState& h = ctx->h_st[0];
    memcpy(out, h.emit, sizeof(int) * h.n_emit);
    *n_out = h.n_emit;
    return LA_OK;
}

extern "C" int la_step_batch(la_ctx* ctx, int32_t* out, int cap, int* n_out)
{
    if (!ctx) return LA_ERR_ARG;
    if (!out || !n_out || cap < ctx->N) return fail(ctx, LA_ERR_ARG, "out must hold N tokens per sequence");
    const int rc = run_step(ctx);
    if (rc) return rc;
    for (int b = 0; b < ctx->B; b++) {
        const DState& h = ctx->h_st[b];
        memcpy(out + (size_t)b * cap, h.emit, sizeof(int) * h.n_emit);
        n_out[b] = h.n_emit;
    }
    return LA_OK;
}

extern "C" int la_set_sampling(la_ctx* ctx, float temperature, uint64_t seed)
{
    if (!ctx) return LA_ERR_ARG;
    if (temperature != temperature || temperature > 3.0e38f) return fail(ctx, LA_ERR_ARG, "temperature must be finite");
    ctx->tau = temperature > 0.f ? temperature : 0.f;
    // sequence b of a batch draws from the stream seeded with seed + b
    std::vector<unsigned long long> v(ctx->B);
    for (int b = 0; b < ctx->B; b++) {
        v[b] = seed + (uint64_t)b;
        LA_CK(cudaMemcpyAsync(&seq_ptr(ctx->st, ctx->sb, b)->rng, &v[b], sizeof(v[b]), cudaMemcpyHostToDevice, ctx->s));
    }
    LA_CK(cudaStreamSynchronize(ctx->s));  // v is a host temporary
    if (ctx->gexec) {  // the step's launch sequence changes: capture it again
        cudaGraphExecDestroy(ctx->gexec);
        ctx->gexec = nullptr;
        cudaGraphDestroy(ctx->graph);
        ctx->graph = nullptr;
    }
    return LA_OK;
}

extern "C" int la_set_top_k(la_ctx* ctx, int top_k)
{
    if (!ctx) return LA_ERR_ARG;
    if (top_k < 0) return fail(ctx, LA_ERR_ARG, "top_k must be >= 0");
    if (top_k != ctx->top_k && ctx->gexec) {  // the step's launches change: capture it again
        cudaGraphExecDestroy(ctx->gexec);
        ctx->gexec = nullptr;
        cudaGraphDestroy(ctx->graph);
        ctx->graph = nullptr;
    }
    ctx->top_k = top_k;
    return LA_OK;
}

extern "C" int la_set_top_p(la_ctx* ctx, float top_p)
{
    if (!ctx) return LA_ERR_ARG;
    if (!(top_p > 0.f && top_p <= 1.f)) return fail(ctx, LA_ERR_ARG, "top_p must be in (0, 1]");
    // floor(top_p 2^24), at least 1 (exact: a float times 2^24 in double)
    const double x = (double)top_p * 16777216.0;
    const unsigned int p24 = top_p >= 1.f ? 1u << 24 : (x < 1.0 ? 1u : (unsigned int)x);
    if (p24 != ctx->top_p24 && ctx->gexec) {  // the step's launches change: capture it again
        cudaGraphExecDestroy(ctx->gexec);
        ctx->gexec = nullptr;
        cudaGraphDestroy(ctx->graph);
        ctx->graph = nullptr;
    }
    ctx->top_p24 = p24;
    return LA_OK;
}

extern "C" int la_generate(la_ctx* ctx, const int32_t* prompt, int len, int max_new, int32_t* out, int* n_out)
{
    if (!ctx) return LA_ERR_ARG;
    if (max_new < 0 || !n_out || (max_new > 0 && !out)) return fail(ctx, LA_ERR_ARG, "bad output buffer");
    int rc = la_prefill(ctx, prompt, len);
    if (rc) return rc;
    int n = 0;
    int32_t buf[kMaxN];
    while (n < max_new) {
        int k = 0;
        rc = la_step(ctx, buf, kMaxN, &k);
        if (rc) break;
        for (int i = 0; i < k && n < max_new; i++) out[n++] = buf[i];
    }
    *n_out = n;
    return rc;
}

extern "C" int la_generate_batch(la_ctx* ctx, const int32_t* prompts, const int* lens, int max_new, int32_t* out,
                                 int* n_out)
{
    if (!ctx) return LA_ERR_ARG;
    if (!prompts || !lens || !n_out || max_new < 0 || (max_new > 0 && !out))
        return fail(ctx, LA_ERR_ARG, "bad prompt or output buffer");
    const int B = ctx->B;
    size_t off = 0;
    for (int b = 0; b < B; b++) {
        if (lens[b] < 1) return fail(ctx, LA_ERR_ARG, "prompt must hold at least one token");
        const int rc = prefill_seq(ctx, b, prompts + off, lens[b]);
        if (rc) return rc;
        off += (size_t)lens[b];
    }
    for (int b = 0; b < B; b++) n_out[b] = 0;
    std::vector<int32_t> buf((size_t)B * kMaxN);
    std::vector<int> n(B);
    int rc = LA_OK;
    auto done = [&]() {
        for (int b = 0; b < B; b++)
            if (n_out[b] < max_new) return false;
        return true;
    };
    // the batch steps every sequence together; a sequence that has its
    // tokens keeps stepping with the others and its further tokens are dropped
    while (!done()) {
        rc = run_step(ctx);
        if (rc) break;
        for (int b = 0; b < B; b++) {
            const DState& h = ctx->h_st[b];
            for (int i = 0; i < h.n_emit && n_out[b] < max_new; i++) out[(size_t)b * max_new + n_out[b]++] = h.emit[i];
        }
    }
    return rc;
}

extern "C" int la_get_profile(la_ctx* ctx, la_prof_entry* out, int cap, int* n_out)
{
    static const char* names[P_NCLS] = {"gemm_qkv", "gemm_o",    "gemm_gateup", "gemm_down", "gemm_lmhead",
                                        "gemm_epilogue", "attention", "rmsnorm", "control"};
    if (!ctx || !out || !n_out) return LA_ERR_ARG;
    if (!ctx->prof.on) return fail(ctx, LA_ERR_STATE, "context made without LA_PROFILE");
    int n = 0;
    for (int c = 0; c < P_NCLS && n < cap; c++) {
        if (!ctx->prof.n[c]) continue;
        la_prof_entry& e = out[n++];
        memset(&e, 0, sizeof(e));
        snprintf(e.name, sizeof(e.name), "%s", names[c]);
        e.launches = ctx->prof.n[c];
        e.total_ms = ctx->prof.ms[c];
        e.bytes = ctx->prof.bytes[c];
        e.flops = ctx->prof.flops[c];
    }
    *n_out = n;
    return LA_OK;
}

extern "C" int la_get_stats(la_ctx* ctx, la_stats* out)
{
    if (!ctx || !out) return LA_ERR_ARG;
    *out = ctx->stats;
    return LA_OK;
}

extern "C" int la_debug_logits(la_ctx* ctx, float* host, size_t n)
{
    if (!ctx || !host) return LA_ERR_ARG;
    if (!ctx->have_step) return fail(ctx, LA_ERR_STATE, "no step yet");
    if (!(ctx->flags & LA_DEBUG_LOGITS)) return fail(ctx, LA_ERR_STATE, "context made without LA_DEBUG_LOGITS");
    size_t need = (size_t)ctx->T * ctx->d.vocab;
    if (n < need) return fail(ctx, LA_ERR_ARG, "buffer too small");
    LA_CK(cudaMemcpyAsync(host, ctx->LOGITS + (size_t)ctx->dseq * need, need * 4, cudaMemcpyDeviceToHost, ctx->s));
    LA_CK(cudaStreamSynchronize(ctx->s));
    return LA_OK;
}

extern "C" int la_debug_argmax(la_ctx* ctx, int32_t* host, int cap, int* T_out)
{
    if (!ctx || !host || !T_out) return LA_ERR_ARG;
    if (!ctx->have_step) return fail(ctx, LA_ERR_STATE, "no step yet");
    if (cap < ctx->T) return fail(ctx, LA_ERR_ARG, "buffer too small");
    LA_CK(cudaMemcpyAsync(host, ctx->AMAX + (size_t)ctx->dseq * ctx->T, (size_t)ctx->T * 4, cudaMemcpyDeviceToHost,
                          ctx->s));
    LA_CK(cudaStreamSynchronize(ctx->s));
    *T_out = ctx->T;
    return LA_OK;
}

extern "C" int la_debug_rows(la_ctx* ctx, int32_t* tok, int32_t* pos, int cap, int* T_out, int* ncand)
{
    if (!ctx || !tok || !pos || !T_out || !ncand) return LA_ERR_ARG;
    if (!ctx->have_step) return fail(ctx, LA_ERR_STATE, "no step yet");
    if (cap < ctx->T) return fail(ctx, LA_ERR_ARG, "buffer too small");
    const size_t r0 = (size_t)ctx->dseq * ctx->T;
    LA_CK(cudaMemcpyAsync(tok, ctx->tok + r0, (size_t)ctx->T * 4, cudaMemcpyDeviceToHost, ctx->s));
    LA_CK(cudaMemcpyAsync(pos, ctx->pos + r0, (size_t)ctx->T * 4, cudaMemcpyDeviceToHost, ctx->s));
    LA_CK(cudaStreamSynchronize(ctx->s));
    *T_out = ctx->T;
    *ncand = ctx->h_st[ctx->dseq].ncand;
    return LA_OK;
}

extern "C" int la_debug_pool(la_ctx* ctx, int32_t key, int32_t* host, int cap, int* count)
{
    if (!ctx || !host || !count) return LA_ERR_ARG;
    const int n1 = ctx->N - 1, tot = (ctx->G > 0 ? ctx->G : 1) * n1;
    if (cap < tot) return fail(ctx, LA_ERR_ARG, "buffer too small");
    if (ctx->G == 0) {
        *count = 0;
        return LA_OK;
    }
    int* dkey = ctx->dbg;
    int* dcnt = ctx->dbg + 1;
    int* dout = ctx->dbg + 2;
    LA_CK(cudaMemcpyAsync(dkey, &key, 4, cudaMemcpyHostToDevice, ctx->s));
    launch_pool_lookup(ctx->s, seq_pool(ctx->pool, ctx->sb, ctx->dseq), dkey, 1, dout, dcnt);
    LA_CK(cudaMemcpyAsync(host, dout, (size_t)tot * 4, cudaMemcpyDeviceToHost, ctx->s));
    LA_CK(cudaMemcpyAsync(count, dcnt, 4, cudaMemcpyDeviceToHost, ctx->s));
    LA_CK(cudaStreamSynchronize(ctx->s));
    return LA_OK;
}

extern "C" int la_debug_set_argmax_override(la_ctx* ctx, const int32_t* host, int n)
{
    if (!ctx) return LA_ERR_ARG;
    if (host && n != ctx->T) return fail(ctx, LA_ERR_ARG, "the override needs one argmax per step row");
    std::vector<int> buf((size_t)ctx->T + 1, 0);
    if (host) {
        for (int i = 0; i < n; i++)
            if (host[i] < 0 || host[i] >= ctx->d.vocab) return fail(ctx, LA_ERR_ARG, "token id out of range");
        buf[0] = 1;
        memcpy(buf.data() + 1, host, (size_t)n * 4);
    }
    LA_CK(cudaMemcpyAsync(seq_ptr(ctx->AOVR, ctx->sb, ctx->dseq), buf.data(), buf.size() * 4, cudaMemcpyHostToDevice,
                          ctx->s));
    LA_CK(cudaStreamSynchronize(ctx->s));  // buf is a host temporary
    return LA_OK;
}

extern "C" int la_debug_select(la_ctx* ctx, int seq)
{
    if (!ctx) return LA_ERR_ARG;
    if (seq < 0 || seq >= ctx->B) return fail(ctx, LA_ERR_ARG, "seq out of range");
    ctx->dseq = seq;
    return LA_OK;
}

extern "C" int la_debug_window(la_ctx* ctx, int32_t* host, int cap)
{
    if (!ctx || !host) return LA_ERR_ARG;
    const int n = (ctx->N - 1) * ctx->W;
    if (cap < n) return fail(ctx, LA_ERR_ARG, "buffer too small");
    if (n) {
        LA_CK(cudaMemcpyAsync(host, seq_ptr(ctx->win, ctx->sb, ctx->dseq), (size_t)n * 4, cudaMemcpyDeviceToHost,
                              ctx->s));
        LA_CK(cudaStreamSynchronize(ctx->s));
    }
    return LA_OK;
}

// ------------------------------------------------------ standalone attention ---

// Device scratch of one la_attention call: row tables, positions, the
// decode state (P) and the split partials.
struct AttnScratch {
    int *rel, *grp, *map, *groups, *pos;
    DState* st;
    float* part;
};

static size_t attn_scratch_bytes(const StepTables& tb, int H, int hd, int max_seq)
{
    return (size_t)(5 * kRows + 1 + tb.map.size()) * 4 + 256 + sizeof(DState) + 256 +
           attn_mma_partial_bytes(H, hd, max_seq);
}

static AttnScratch attn_scratch_carve(char* base, const StepTables& tb)
{
    AttnScratch a;
    int* ip = (int*)base;
    a.rel = ip;
    a.grp = ip + kRows;
    a.groups = ip + 2 * kRows;          // 2 * kRows + 1
    a.pos = ip + 4 * kRows + 1;
    a.map = ip + 5 * kRows + 1;
    size_t off = ((size_t)(5 * kRows + 1 + tb.map.size()) * 4 + 255) & ~(size_t)255;
    a.st = (DState*)(base + off);
    off += (sizeof(DState) + 255) & ~(size_t)255;
    a.part = (float*)(base + off);
    return a;
}

// Checks shared by la_attention and its no-allocation variant; fills tb.
static int attn_check(int H, int Hkv, int hd, int max_seq, int P, int W, int N, int G, StepTables* tb)
{
    if ((hd != 64 && hd != 128) || H < 1 || Hkv < 1 || H % Hkv) return LA_ERR_ARG;
    if (W < 0 || G < 0 || N < 2 || N > kMaxN || step_rows(W, N, G) > kRows || (N - 1) * W > 127) return LA_ERR_ARG;
    *tb = step_tables(W, N, G);
    if (P < 0 || P + tb->maxoff > max_seq) return LA_ERR_CAPACITY;
    return LA_OK;
}

// One-time kernel set-up (dynamic shared-memory limit) of the standalone
// attention ops, per device and head_dim: cudaFuncSetAttribute applies to
// the current device only.  Thread-safe.
static std::mutex g_attn_init_mu;
static unsigned char g_attn_ready[256][2];

static int attn_ready(int hd)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_attn_init_mu);
    unsigned char& done = g_attn_ready[dev][hd == 128 ? 1 : 0];
    if (!done) {
        if (!attn_mma_init(hd)) return LA_ERR_CUDA;
        done = 1;
    }
    return LA_OK;
}

// Launch the step attention on device tables and scratch, wait for it and
// return its status.
static int attn_launch_sync(DState* st, RowSet rs, int max_rel, const int* pos, const void* q, const void* k_cache,
                            const void* v_cache, const void* k_step, const void* v_step, void* out, float* part, int T,
                            int H, int Hkv, int hd, int max_seq, cudaStream_t s)
{
    launch_attn_mma(s, st, rs, max_rel, pos, q, k_cache, v_cache, k_step, v_step, out, part, T, H, Hkv, hd, max_seq);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

// Upload the tables and launch; scratch is device memory of attn_scratch_bytes.
static int attn_run(const StepTables& tb, char* scratch, const void* q, const void* k_cache, const void* v_cache,
                    const void* k_step, const void* v_step, void* out, int H, int Hkv, int hd, int max_seq, int P,
                    cudaStream_t s)
{
    if (int rc = attn_ready(hd)) return rc;
    AttnScratch a = attn_scratch_carve(scratch, tb);
    std::vector<int> pos(kRows, P);
    for (int r = 0; r < tb.T; r++) pos[r] = P + tb.rel[r];
    DState hst{};
    hst.P = P;
    hst.T = tb.T;
    hst.ncand = 0;
    if (cudaMemcpyAsync(a.rel, tb.rel.data(), kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(a.grp, tb.grp.data(), kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(a.groups, tb.groups.data(), tb.groups.size() * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(a.pos, pos.data(), kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(a.map, tb.map.data(), tb.map.size() * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(a.st, &hst, sizeof(DState), cudaMemcpyHostToDevice, s))
        return LA_ERR_CUDA;
    RowSet rs{a.rel, a.grp, a.map, a.groups, a.groups + kRows + 1, tb.maxoff, tb.ngrp};
    // synchronises: the host tables above are pageable
    return attn_launch_sync(a.st, rs, tb.maxoff - 1, a.pos, q, k_cache, v_cache, k_step, v_step, out, a.part, tb.T, H,
                            Hkv, hd, max_seq, s);
}

extern "C" int la_attention(const void* q, const void* k_cache, const void* v_cache, const void* k_step,
                            const void* v_step, void* out, int n_heads, int n_kv_heads, int head_dim, int max_seq,
                            int P, int W, int N, int G, void* stream)
{
    if (!q || !k_cache || !v_cache || !k_step || !v_step || !out) return LA_ERR_ARG;
    StepTables tb;
    int rc = attn_check(n_heads, n_kv_heads, head_dim, max_seq, P, W, N, G, &tb);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t bytes = attn_scratch_bytes(tb, n_heads, head_dim, max_seq);
    char* scratch = nullptr;
    if (cudaMallocAsync((void**)&scratch, bytes, s) != cudaSuccess) return LA_ERR_OOM;
    rc = attn_run(tb, scratch, q, k_cache, v_cache, k_step, v_step, out, n_heads, n_kv_heads, head_dim, max_seq, P,
                  s);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

// ------------------------------------------ attention without allocation ---
//
// For callers that must not allocate device memory: runtimes that take all
// device memory into one pool at start-up and forbid further allocation, and
// latency-bound callers that cannot accept cudaMalloc's implicit device-wide
// synchronisation.  The scratch lives in one file-scope device array that
// every GPU loading this library holds until the process exits.  No
// cudaMalloc/cudaFree and no host heap: the row tables are built in a
// fixed-size per-thread buffer.

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[256];  // device address of the array, per device ordinal

// Host code may not use the array's name as an address: look its device
// address up once per device, with that device current.
static int noalloc_scratch(char** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = (char*)g_noalloc_ptr[dev];
    return LA_OK;
}

// Fixed-size copy of the step tables (same content as step_tables() for the
// column mask; the standalone attention has no diagonal-levels option).
struct FixedTables {
    int T, maxoff, ngrp;
    int rel[kRows], grp[kRows], groups[2 * kRows + 1], pos[kRows];
    int map[kRows * kRows];
};

static int fixed_tables(int W, int N, int G, int P, FixedTables* tb)
{
    const int n1 = N - 1;
    tb->T = step_rows(W, N, G);
    for (int r = 0; r < kRows; r++) tb->rel[r] = tb->grp[r] = 0;
    for (int l = 0; l < n1; l++)
        for (int j = 0; j < W; j++) {
            tb->rel[1 + l * W + j] = 1 + j + l;
            tb->grp[1 + l * W + j] = j;
        }
    for (int g = 0; g < G; g++)
        for (int i = 0; i < n1; i++) {
            tb->rel[1 + W * n1 + g * n1 + i] = 1 + i;
            tb->grp[1 + W * n1 + g * n1 + i] = W + g;
        }
    tb->maxoff = 1;
    for (int r = 0; r < tb->T; r++) tb->maxoff = tb->rel[r] + 1 > tb->maxoff ? tb->rel[r] + 1 : tb->maxoff;
    tb->ngrp = W + G > 0 ? W + G : 1;
    for (int i = 0; i < tb->ngrp * tb->maxoff; i++) tb->map[i] = 0;
    for (int j = 0; j < W; j++) {
        int* m = &tb->map[j * tb->maxoff];
        for (int jj = 0; jj <= j; jj++) m[1 + jj] = 1 + jj;
        for (int l = 1; l < n1; l++) m[1 + j + l] = 1 + l * W + j;
    }
    for (int g = 0; g < G; g++)
        for (int i = 0; i < n1; i++) tb->map[(W + g) * tb->maxoff + 1 + i] = 1 + W * n1 + g * n1 + i;
    int k = 0;
    for (int g = 0; g < tb->ngrp; g++) {
        tb->groups[g] = k;
        for (int r = 0; r < tb->T; r++)
            if (tb->grp[r] == g) tb->groups[kRows + 1 + k++] = r;
    }
    tb->groups[tb->ngrp] = k;
    for (int r = 0; r < kRows; r++) tb->pos[r] = P + (r < tb->T ? tb->rel[r] : 0);
    return LA_OK;
}

extern "C" int la_attention_noalloc(const void* q, const void* k_cache, const void* v_cache, const void* k_step,
                                    const void* v_step, void* out, int n_heads, int n_kv_heads, int head_dim,
                                    int max_seq, int P, int W, int N, int G, void* stream)
{
    if (!q || !k_cache || !v_cache || !k_step || !v_step || !out) return LA_ERR_ARG;
    if ((head_dim != 64 && head_dim != 128) || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads) return LA_ERR_ARG;
    if (W < 0 || G < 0 || N < 2 || N > kMaxN || step_rows(W, N, G) > kRows || (N - 1) * W > 127) return LA_ERR_ARG;
    static thread_local FixedTables tb;  // 66 KB: kept off the stack, no heap
    fixed_tables(W, N, G, P, &tb);
    if (P < 0 || P + tb.maxoff > max_seq) return LA_ERR_CAPACITY;
    // scratch layout: rel | grp | groups | pos | map | state | split partials
    const size_t tables = ((size_t)(5 * kRows + 1 + tb.ngrp * tb.maxoff) * 4 + 255) & ~(size_t)255;
    const size_t state = (sizeof(DState) + 255) & ~(size_t)255;
    const size_t need = tables + state + attn_mma_partial_bytes(n_heads, head_dim, max_seq);
    if (need > kNoAllocScratchBytes) {
        fprintf(stderr, "la_attention_noalloc: needs %zu bytes of scratch, the fixed array holds %zu\n", need,
                kNoAllocScratchBytes);
        return LA_ERR_CAPACITY;
    }
    char* base = nullptr;
    int rc = noalloc_scratch(&base);
    if (rc) return rc;
    if ((rc = attn_ready(head_dim))) return rc;
    int* ip = (int*)base;
    DState* st = (DState*)(base + tables);
    float* part = (float*)(base + tables + state);
    DState hst{};
    hst.P = P;
    hst.T = tb.T;
    cudaStream_t s = (cudaStream_t)stream;
    // every piece the kernels read is rewritten here; the partials are
    // written before they are read, so nothing needs clearing
    if (cudaMemcpyAsync(ip, tb.rel, kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(ip + kRows, tb.grp, kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(ip + 2 * kRows, tb.groups, (2 * kRows + 1) * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(ip + 4 * kRows + 1, tb.pos, kRows * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(ip + 5 * kRows + 1, tb.map, (size_t)tb.ngrp * tb.maxoff * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(st, &hst, sizeof(DState), cudaMemcpyHostToDevice, s))
        return LA_ERR_CUDA;
    RowSet rs{ip, ip + kRows, ip + 5 * kRows + 1, ip + 2 * kRows, ip + 3 * kRows + 1, tb.maxoff, tb.ngrp};
    // synchronises: the host tables are reused by the next call on this thread
    return attn_launch_sync(st, rs, tb.maxoff - 1, ip + 4 * kRows + 1, q, k_cache, v_cache, k_step, v_step, out, part,
                            tb.T, n_heads, n_kv_heads, head_dim, max_seq, s);
}

// --------------------------------------------------------- standalone pool ---

struct la_pool {
    PoolView v;
    cudaStream_t s;
    int* mem;
    int* status;
    int max_bulk;
};

extern "C" int la_pool_create(int capacity, int N, int G, void* stream, la_pool** out)
{
    if (!out) return LA_ERR_ARG;
    *out = nullptr;
    if (capacity < 1 || N < 2 || N > kMaxN || G < 1 || G * (N - 1) > 1024) return LA_ERR_ARG;
    int lg = next_pow2_log2(capacity < 64 ? 64 : capacity);
    if (lg > 28) return LA_ERR_ARG;
    const size_t cap = (size_t)1 << lg;
    const int max_bulk = 1 << 22;
    la_pool* p = new (std::nothrow) la_pool();
    if (!p) return LA_ERR_OOM;
    size_t ints = cap * 3 + cap * (size_t)G * (N - 1) + max_bulk + 1;
    if (cudaMalloc((void**)&p->mem, ints * 4) != cudaSuccess) {
        delete p;
        return LA_ERR_OOM;
    }
    int* m = p->mem;
    p->status = m + ints - 1;
    p->v = PoolView{m, m + cap, m + 3 * cap, m + 2 * cap, m + 3 * cap + cap * (size_t)G * (N - 1), p->status,
                    (int)cap, lg, G, N - 1};
    p->s = (cudaStream_t)stream;
    p->max_bulk = max_bulk;
    launch_pool_reset(p->s, p->v);
    if (cudaMemsetAsync(p->status, 0, 4, p->s) != cudaSuccess || cudaStreamSynchronize(p->s) != cudaSuccess) {
        cudaFree(p->mem);
        delete p;
        return LA_ERR_CUDA;
    }
    *out = p;
    return LA_OK;
}

extern "C" int la_pool_insert(la_pool* p, const int32_t* keys, const int32_t* grams, int n)
{
    if (!p || n < 0 || (n > 0 && (!keys || !grams))) return LA_ERR_ARG;
    if (n > p->max_bulk) return LA_ERR_ARG;
    if (cudaMemsetAsync(p->status, 0, 4, p->s) != cudaSuccess) return LA_ERR_CUDA;
    launch_pool_insert(p->s, p->v, keys, grams, p->v.n1, n);
    int st = 0;
    if (cudaMemcpyAsync(&st, p->status, 4, cudaMemcpyDeviceToHost, p->s) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaStreamSynchronize(p->s) != cudaSuccess) return LA_ERR_CUDA;
    return st;  // LA_OK, LA_ERR_CAPACITY (table full) or LA_ERR_ARG (a negative key)
}

extern "C" int la_pool_lookup(la_pool* p, const int32_t* keys, int n, int32_t* out, int32_t* counts)
{
    if (!p || n < 0 || (n > 0 && (!keys || !out || !counts))) return LA_ERR_ARG;
    launch_pool_lookup(p->s, p->v, keys, n, out, counts);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

extern "C" int la_pool_size(la_pool* p, int* n_keys)
{
    if (!p || !n_keys) return LA_ERR_ARG;
    std::vector<int> k(p->v.cap);
    if (cudaMemcpyAsync(k.data(), p->v.keys, (size_t)p->v.cap * 4, cudaMemcpyDeviceToHost, p->s) != cudaSuccess)
        return LA_ERR_CUDA;
    if (cudaStreamSynchronize(p->s) != cudaSuccess) return LA_ERR_CUDA;
    int c = 0;
    for (int x : k) c += (x != -1);
    *n_keys = c;
    return LA_OK;
}

extern "C" void la_pool_destroy(la_pool* p)
{
    if (!p) return;
    cudaStreamSynchronize(p->s);
    cudaFree(p->mem);
    delete p;
}
