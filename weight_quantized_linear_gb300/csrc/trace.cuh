// trace.cuh -- phase stamps for a developer build of the library.
//
// Compiled in only with -DWQL_PHASE_TRACE (build.build(trace=True) writes that build to a library
// file of its own; the library the package loads by default never defines the macro, and there
// every macro below expands to nothing).  At fixed phase points of a kernel one thread of a CTA
// writes %globaltimer into its row of kTraceSlots stamps.  The row is picked by the launch -- the
// offset of the kernel's output pointer from a registered base, in units of a registered stride,
// so that a harness giving every launch its own output buffer tells the launches apart -- and by
// the CTA's linear index.  The stamps add stores only: no work is skipped or reordered.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace wql {

constexpr int kTraceSlots = 32;

struct TraceDesc {
  unsigned long long* buf;        // [launches][ctas][kTraceSlots] ns, zero where nothing stamped
  unsigned long long ybase;       // output pointer of launch 0
  unsigned long long ystride;     // bytes between the output pointers of consecutive launches
  int launches, ctas;
};

#ifdef WQL_PHASE_TRACE
// One copy per translation unit (the library is compiled without relocatable device code):
// each traced source file registers the descriptor with its own trace_set_local().
static __device__ TraceDesc g_trace_desc;

__device__ __forceinline__ unsigned long long* trace_row(const void* y) {
  const TraceDesc d = g_trace_desc;
  const unsigned long long a = reinterpret_cast<unsigned long long>(y);
  if (d.buf == nullptr || d.ystride == 0 || a < d.ybase) return nullptr;
  const unsigned long long l = (a - d.ybase) / d.ystride;
  const unsigned long long cta = blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (l >= (unsigned long long)d.launches || cta >= (unsigned long long)d.ctas) return nullptr;
  return d.buf + (l * d.ctas + cta) * kTraceSlots;
}

static inline cudaError_t trace_set_local(const TraceDesc& d) {
  return cudaMemcpyToSymbol(g_trace_desc, &d, sizeof(d));
}

#define WQL_TRACE_ROW(y) unsigned long long* const wql_trace_row_ = ::wql::trace_row(y)
#define WQL_STAMP(slot)                                                     \
  do {                                                                      \
    if (wql_trace_row_) wql_trace_row_[(slot)] = ::wql::globaltimer_ns();   \
  } while (0)
// the latest of several threads' stamps
#define WQL_STAMP_MAX(slot)                                                            \
  do {                                                                                 \
    if (wql_trace_row_) atomicMax(&wql_trace_row_[(slot)], ::wql::globaltimer_ns());   \
  } while (0)
// the SM the CTA runs on, in the last slot
#define WQL_STAMP_SMID()                                                  \
  do {                                                                    \
    if (wql_trace_row_) {                                                 \
      unsigned smid_;                                                     \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                  \
      wql_trace_row_[kTraceSlots - 1] = smid_;                            \
    }                                                                     \
  } while (0)
#else
#define WQL_TRACE_ROW(y) \
  do {                   \
  } while (0)
#define WQL_STAMP(slot) \
  do {                  \
  } while (0)
#define WQL_STAMP_MAX(slot) \
  do {                      \
  } while (0)
#define WQL_STAMP_SMID() \
  do {                   \
  } while (0)
#endif

}  // namespace wql
