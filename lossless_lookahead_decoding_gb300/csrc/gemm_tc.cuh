// gemm_tc.cuh -- tensor-core (tcgen05/TMEM, TMA-fed) path of the bf16 decoder
// forward: the projection/MLP/LM-head GEMMs with fused epilogues and the
// masked attention.
#pragma once
#include <cuda_runtime.h>

#include "../../include/lookahead.h"
#include "common.cuh"

namespace la {

struct TcPlan {
    bool ok = false;
    void* impl = nullptr;        // owned state (tensor maps, split-K scratch)
    Profiler* prof = nullptr;    // optional kernel timing
    int carveout = -1;           // >= 0: preferred shared-memory carveout (%) of every launch
};

// 0 = plan made, 1 = shape not supported (caller falls back to SIMT), < 0 error.
// status: device word that bounded waits set to LA_ERR_TIMEOUT on give-up.
int tc_plan_create(TcPlan* p, const la_model_desc& d, const void* const* lw, void* XN, void* Q, void* ATT, void* HID,
                   int esz, int* status);
void tc_plan_destroy(TcPlan* p);
void tc_qkv_rope(const TcPlan& p, cudaStream_t s, int layer, int rows, const int* pos, const float* cosb,
                 const float* sinb, void* Q, void* KS, void* VS);
// O-proj / down GEMMs whose residual add is left pending, to be folded into
// the RMSNorm that follows (tc_resid_rmsnorm): X += partial sums, XN = norm(X).
struct TcResid {
    int tiles, KB, ctas, rows;
    const float* partial;
};
TcResid tc_oproj(const TcPlan& p, cudaStream_t s, int layer, int rows);
TcResid tc_down(const TcPlan& p, cudaStream_t s, int layer, int rows);
void tc_resid_rmsnorm(const TcPlan& p, cudaStream_t s, const TcResid& pend, float* X, const void* w, void* XN, int d,
                      float eps);
void tc_gateup_swiglu(const TcPlan& p, cudaStream_t s, int layer, int rows);
void tc_lmhead_argmax(const TcPlan& p, cudaStream_t s, int rows, float* logits, unsigned long long* amaxp, int* amax);

}  // namespace la
