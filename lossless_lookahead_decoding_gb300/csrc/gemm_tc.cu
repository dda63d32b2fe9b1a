// gemm_tc.cu -- placeholder until the tcgen05 kernels land: reports every
// shape as unsupported so bf16 models run on the SIMT kernels.
#include "gemm_tc.cuh"

namespace la {

int tc_plan_create(TcPlan* p, const la_model_desc&, const void* const*, void*, void*, void*, void*, int)
{
    p->ok = false;
    return 1;
}
void tc_plan_destroy(TcPlan* p) { p->ok = false; }
void tc_qkv_rope(const TcPlan&, cudaStream_t, int, int, const int*, const float*, const float*, void*, void*, void*) {}
bool tc_attn_supported(const TcPlan&) { return false; }
void tc_attention(const TcPlan&, cudaStream_t, const DState*, const RowSet&, const int*, const void*, const void*,
                  const void*, const void*, const void*, void*, int) {}
void tc_oproj_resid(const TcPlan&, cudaStream_t, int, int, float*) {}
void tc_gateup_swiglu(const TcPlan&, cudaStream_t, int, int) {}
void tc_down_resid(const TcPlan&, cudaStream_t, int, int, float*) {}
void tc_lmhead_argmax(const TcPlan&, cudaStream_t, int, float*, unsigned long long*, int*) {}

}  // namespace la
