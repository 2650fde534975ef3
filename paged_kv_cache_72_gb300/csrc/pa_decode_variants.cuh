// Kernel-variant dispatch for one head_dim and one KV element type; included
// by pa_decode_d64.cu, pa_decode_d128.cu (16-bit caches) and
// pa_decode_f8_d64.cu, pa_decode_f8_d128.cu (E4M3 caches), so that they
// compile in parallel.
#pragma once

#include "pa_decode_kernel.cuh"
#include "pa_decode_launch.h"

namespace pa {

template <int D, bool BF, int MODE, bool SWZ, bool HI, bool F8>
struct Variant {
  static decltype(&paged_decode_kernel<D, BF, MODE, SWZ, HI, F8>) fn() {
    return &paged_decode_kernel<D, BF, MODE, SWZ, HI, F8>;
  }
};

// Calls f(kernel_pointer) for the variant the plan selects (kF8: the plan is
// for an E4M3 cache; its TU instantiates only those variants).
template <int D, bool kF8, class F>
int with_variant(const DecodePlan& p, F&& f) {
  if constexpr (kF8) {
#define PA_V8(BF, MODE, SWZ, HI) return f(Variant<D, BF, MODE, SWZ, HI, true>::fn())
    if (p.mode == kModeSimt) {
      if (p.bf16) PA_V8(true, kModeSimt, false, false);
      PA_V8(false, kModeSimt, false, false);
    }
    if (p.bf16) {
      if (p.swz) {
        if (p.hi) PA_V8(true, kModeMma, true, true);
        PA_V8(true, kModeMma, true, false);
      }
      if (p.hi) PA_V8(true, kModeMma, false, true);
      PA_V8(true, kModeMma, false, false);
    }
    if (p.swz) {
      if (p.hi) PA_V8(false, kModeMma, true, true);
      PA_V8(false, kModeMma, true, false);
    }
    if (p.hi) PA_V8(false, kModeMma, false, true);
    PA_V8(false, kModeMma, false, false);
#undef PA_V8
  } else {
#define PA_V(BF, MODE, SWZ, HI) return f(Variant<D, BF, MODE, SWZ, HI, false>::fn())
  if (p.mode == kModeSimt) {
    if (p.bf16) PA_V(true, kModeSimt, false, false);
    PA_V(false, kModeSimt, false, false);
  }
  if (p.mode == kModeGather) {
    if (p.bf16) {
      if (p.swz) PA_V(true, kModeGather, true, false);
      PA_V(true, kModeGather, false, false);
    }
    if (p.swz) PA_V(false, kModeGather, true, false);
    PA_V(false, kModeGather, false, false);
  }
  if (p.bf16) {
    if (p.swz) {
      if (p.hi) PA_V(true, kModeMma, true, true);
      PA_V(true, kModeMma, true, false);
    }
    if (p.hi) PA_V(true, kModeMma, false, true);
    PA_V(true, kModeMma, false, false);
  }
  if (p.swz) {
    if (p.hi) PA_V(false, kModeMma, true, true);
    PA_V(false, kModeMma, true, false);
  }
  if (p.hi) PA_V(false, kModeMma, false, true);
  PA_V(false, kModeMma, false, false);
#undef PA_V
  }
}

// Opt the variant in to the device's full shared memory (one kernel serves
// plans of different sizes, so the limit is the device maximum, not this
// plan's size) and report resident CTAs per SM for this plan.
template <int D, bool kF8>
int ctas_per_sm_impl(const DecodePlan& p, int* ctas) {
  return with_variant<D, kF8>(p, [&](auto kern) -> int {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         p.smem_optin);
    if (e != cudaSuccess) return launch_status(e, "cudaFuncSetAttribute");
    if (split_regs(p.mode, kF8, p.hi)) {
      // the warpgroups re-divide the registers the block is launched with;
      // with fewer at launch the consumers' request could not be met
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return launch_status(e, "cudaFuncGetAttributes");
      if (fa.numRegs < kLaunchRegs) return PA_ERR_UNSUPPORTED;
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, block_threads(p.mode, kF8, p.hi),
                                                      p.smem_bytes);
    if (e != cudaSuccess) return launch_status(e, "occupancy query");
    *ctas = n;
    return PA_OK;
  });
}

template <int D, bool kF8>
int launch_impl(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                const DecodeArgs& a, cudaStream_t s) {
  clear_stale_error();
  // no CTA waits for another, so any grid size runs as an ordinary launch
  return with_variant<D, kF8>(p, [&](auto kern) -> int {
    const cudaError_t e =
        launch_pdl(kern, dim3(p.grid), dim3(block_threads(p.mode, kF8, p.hi)), (size_t)p.smem_bytes,
                   s, tk, tv, a);
    return launch_status(e, "decode kernel launch");
  });
}

}  // namespace pa
