// The decode kernel instantiations of one head_dim and one merge mode,
// selected when compiling: -DGQA_INST_HD=<64|128|256> -DGQA_INST_CLUSTER=<0|1>.
// Each combination is its own translation unit so that they compile in
// parallel; the host code reaches them through decode_launch.h.
#include "decode_kernel.cuh"
#include "decode_launch.h"

#if !defined(GQA_INST_HD) || !defined(GQA_INST_CLUSTER)
#error "compile with -DGQA_INST_HD=<64|128|256> -DGQA_INST_CLUSTER=<0|1>"
#endif

#define GQA_REF_NAME_(hd, cl) decode_kernel_ref_##hd##_##cl
#define GQA_REF_NAME(hd, cl) GQA_REF_NAME_(hd, cl)

namespace gqa {
namespace {

template <int NP, bool F16>
KernelRef ref() {
  using Cfg = DecodeCfg<GQA_INST_HD, NP>;
  return KernelRef{reinterpret_cast<const void*>(&gqa_decode_kernel<GQA_INST_HD, NP, F16, GQA_INST_CLUSTER != 0>),
                   Cfg::kSmemBytes, Cfg::kThreads};
}

}  // namespace

KernelRef GQA_REF_NAME(GQA_INST_HD, GQA_INST_CLUSTER)(int np, bool f16) {
  if (np <= 16) return f16 ? ref<16, true>() : ref<16, false>();
  return f16 ? ref<32, true>() : ref<32, false>();
}

}  // namespace gqa
