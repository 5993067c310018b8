// large_t.cu -- the layer for prefill-sized batches (T > 8).
#include "layer.cuh"

namespace moe {

int large_t_setup(moe_layer* L, cudaStream_t st) {
  (void)L;
  (void)st;
  return MOE_OK;
}

int large_t_forward(moe_layer* L, const void* x, int T, void* y, cudaStream_t st) {
  (void)L; (void)x; (void)T; (void)y; (void)st;
  return MOE_EINVAL;
}

int large_t_get_routing(moe_layer* L, int32_t* ids, float* gates, int32_t* offsets, int32_t* perm, cudaStream_t st) {
  (void)L; (void)ids; (void)gates; (void)offsets; (void)perm; (void)st;
  return MOE_EINVAL;
}

void large_t_release(moe_layer* L) { (void)L; }

}  // namespace moe
