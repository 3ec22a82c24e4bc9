// Handles on the decode kernel instantiations, which are compiled in separate
// translation units (decode_instances.cu, once per head_dim and merge mode)
// so that the library builds in parallel.
#pragma once

namespace gqa {

struct KernelRef {
  const void* fn;  // the __global__ function, for cudaLaunchKernelExC / cudaFuncSetAttribute
  int smem_bytes;  // dynamic shared memory it is launched with
  int threads;     // CTA size
};

// np: padded head columns (16 or 32); f16: fp16 inputs (else bf16).
KernelRef decode_kernel_ref_64_0(int np, bool f16);
KernelRef decode_kernel_ref_128_0(int np, bool f16);
KernelRef decode_kernel_ref_256_0(int np, bool f16);
KernelRef decode_kernel_ref_64_1(int np, bool f16);   // in-cluster merge
KernelRef decode_kernel_ref_128_1(int np, bool f16);
KernelRef decode_kernel_ref_256_1(int np, bool f16);

}  // namespace gqa
