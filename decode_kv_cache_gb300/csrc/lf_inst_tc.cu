// Instantiations of the tensor-core (tcgen05) decode kernel: bf16, head_dim 128.
#include "lf_decode_tc.cuh"
#include "lf_kernels.h"

namespace lf {
namespace {

template <int G>
int smem_bytes_tc(int stages, int chunk, int cluster, int evict, int items) {
  return TcPlan<G>::smem_bytes(stages, chunk, cluster, evict, items);
}

template <int G>
bool fill(KernelEntry* e) {
  e->kind = kTensorCore;
  e->decode = reinterpret_cast<const void*>(&decode_step_tc_kernel<G, false>);
  e->decode_split = reinterpret_cast<const void*>(&decode_step_tc_kernel<G, true>);
  e->prefill = reinterpret_cast<const void*>(&prefill_kernel<__nv_bfloat16, 128>);
  e->select = reinterpret_cast<const void*>(&select_layer_kernel<__nv_bfloat16, 128>);
  e->smem_bytes = &smem_bytes_tc<G>;
  e->head_dim = 128;
  e->group = G;
  e->elem_bytes = 2;
  return true;
}

}  // namespace

bool find_kernels_tc(int head_dim, int group, KernelEntry* e) {
  if (head_dim != 128) return false;
  switch (group) {
    case 1: return fill<1>(e);
    case 2: return fill<2>(e);
    case 4: return fill<4>(e);
    case 8: return fill<8>(e);
    default: return false;
  }
}

}  // namespace lf
