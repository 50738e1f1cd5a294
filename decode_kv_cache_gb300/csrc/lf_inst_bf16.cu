// Instantiations of the decode and prefill kernels for bf16 storage.
#include "lf_decode.cuh"
#include "lf_kernels.h"

namespace lf {
namespace {

template <int D, int G>
int smem_bytes_bf16(int stages, int chunk, int /*cluster*/, int /*evict*/, int /*items*/) {
  return DecodePlan<__nv_bfloat16, D, G>::smem_bytes(stages, chunk);
}

template <int D, int G>
bool fill(KernelEntry* e) {
  e->decode = reinterpret_cast<const void*>(&decode_step_simt_kernel<__nv_bfloat16, D, G>);
  e->prefill = reinterpret_cast<const void*>(&prefill_kernel<__nv_bfloat16, D>);
  e->select = reinterpret_cast<const void*>(&select_layer_kernel<__nv_bfloat16, D>);
  e->smem_bytes = &smem_bytes_bf16<D, G>;
  e->head_dim = D;
  e->group = G;
  e->elem_bytes = (int)sizeof(__nv_bfloat16);
  return true;
}

template <int D>
bool by_group(int group, KernelEntry* e) {
  switch (group) {
    case 1: return fill<D, 1>(e);
    case 2: return fill<D, 2>(e);
    case 4: return fill<D, 4>(e);
    case 8: return fill<D, 8>(e);
    default: return false;
  }
}

}  // namespace

bool find_kernels_bf16(int head_dim, int group, KernelEntry* e) {
  switch (head_dim) {
    case 16: return by_group<16>(group, e);
    case 32: return by_group<32>(group, e);
    case 64: return by_group<64>(group, e);
    case 128: return by_group<128>(group, e);
    default: return false;
  }
}

}  // namespace lf
