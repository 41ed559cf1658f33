// Tree-verify attention on the 5th-generation tensor cores (tcgen05): placeholder
// until the kernel lands; the dispatcher then uses the CUDA-core kernel.
#include "attn_common.cuh"

namespace specv {

int attn_splits_tc(int batch, int max_nodes, int hq, int hkv, int max_prefix) {
  return attn_splits_simt(batch, max_nodes, hq, hkv, max_prefix);
}

bool attn_tc_supported(int, int, int, int, int, int) { return false; }

int launch_attn_tc(const void*, const void*, const void*, int, int, const int32_t*, int, const int32_t*, int,
                   const void*, const void*, const uint64_t*, const int32_t*, int, int, int, int, int, int, float,
                   void*, float*, void*, int32_t*, cudaStream_t) {
  return SPEC_ERR_UNSUPPORTED;
}

}  // namespace specv
