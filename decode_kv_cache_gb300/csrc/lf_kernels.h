// Internal table of compiled decode/prefill kernel instantiations.
#pragma once

namespace lf {

struct KernelEntry {
  const void* decode = nullptr;   // __global__ void(DecodeArgs)
  const void* prefill = nullptr;  // __global__ void(PrefillArgs)
  int (*smem_bytes)(int stages, int chunk) = nullptr;
  int head_dim = 0, group = 0, elem_bytes = 0;
};

// Defined in one translation unit per element type.
bool find_kernels_bf16(int head_dim, int group, KernelEntry* out);
bool find_kernels_f32(int head_dim, int group, KernelEntry* out);

}  // namespace lf
