// Device-side kernel spans (tracing aid): per kernel id, the sum over
// launches of %globaltimer from the first CTA past its grid-dependency wait
// to the last warp's exit, and the number of launches.  A kernel inside a
// replayed CUDA graph cannot be bracketed by events; this record can.
//
// Every translation unit that includes this header gets its own record
// (internal linkage); its span_control_* function reads and resets it.  A
// kernel marks its start with span_begin(id) (thread 0 of each CTA, after
// the dependency wait) and declares `SpanExit` at its top, whose destructor
// runs on every return path of every thread: lane 0 of each warp stamps the
// end and counts the warp out; the grid's last warp adds the span to the
// totals and clears the record for the next launch.  Launches of one kernel
// id must not overlap in time (stream order, or a dependency wait before
// span_begin, guarantees it).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds4moe.h"

namespace ds4 {

struct KSpan {
  unsigned long long nbegin;  // ~(earliest start): the zero record means "none yet"
  unsigned long long end, sum_ns;
  unsigned int exited, count;
};

static __device__ KSpan g_spans[DS4MOE_SPAN_COUNT];
static __device__ int g_span_on = 0;

__device__ __forceinline__ unsigned long long span_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void span_begin(int id) {
  if (threadIdx.x == 0 && g_span_on) atomicMax(&g_spans[id].nbegin, ~span_clock());
}

struct SpanExit {
  int id;
  __device__ explicit SpanExit(int i) : id(i) {}
  __device__ ~SpanExit() {
    if ((threadIdx.x & 31u) != 0u || !g_span_on) return;
    KSpan &sp = g_spans[id];
    atomicMax(&sp.end, span_clock());
    __threadfence();
    const unsigned int warps = gridDim.x * gridDim.y * gridDim.z * ((blockDim.x * blockDim.y * blockDim.z) >> 5);
    if (atomicAdd(&sp.exited, 1u) == warps - 1u) {
      __threadfence();
      const unsigned long long nb = atomicExch(&sp.nbegin, 0ull), e = atomicExch(&sp.end, 0ull);
      if (nb != 0ull && e >= ~nb) {
        atomicAdd(&sp.sum_ns, e - ~nb);
        atomicAdd(&sp.count, 1u);
      }
      atomicExch(&sp.exited, 0u);
    }
  }
};

// Host: adds this unit's totals into total_ns[] / launches[] (arrays of
// DS4MOE_SPAN_COUNT, either may be null); with on = 0 / 1 then clears them
// and switches recording off / on.
static inline cudaError_t span_control_unit(int on, double *total_ns, int64_t *launches) {
  KSpan sp[DS4MOE_SPAN_COUNT];
  cudaError_t e = cudaMemcpyFromSymbol(sp, g_spans, sizeof(sp));
  if (e != cudaSuccess) return e;
  for (int i = 0; i < DS4MOE_SPAN_COUNT; ++i) {
    if (total_ns) total_ns[i] += (double)sp[i].sum_ns;
    if (launches) launches[i] += sp[i].count;
  }
  if (on >= 0) {
    const KSpan z[DS4MOE_SPAN_COUNT] = {};
    e = cudaMemcpyToSymbol(g_spans, z, sizeof(z));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_span_on, &on, sizeof(int));
  }
  return e;
}

// One per translation unit with spanned kernels (defined there).
cudaError_t span_control_abi(int on, double *total_ns, int64_t *launches);
cudaError_t span_control_decode(int on, double *total_ns, int64_t *launches);
cudaError_t span_control_t1r(int on, double *total_ns, int64_t *launches);
cudaError_t span_control_prefill(int on, double *total_ns, int64_t *launches);
cudaError_t span_control_shared(int on, double *total_ns, int64_t *launches);

}  // namespace ds4
