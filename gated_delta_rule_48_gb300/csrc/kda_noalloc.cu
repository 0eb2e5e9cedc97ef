// kda_chunk_fwd_noalloc: the prefill without any device allocation.
//
// kda_chunk_fwd takes a small stream-ordered workspace from a memory pool for
// its segment plan (and, when it splits long sequences, for the per-segment
// increment / transition records).  Some callers cannot allow that: runtimes
// that reserve all device memory for their own allocator when they start, or
// callers that must not take allocator locks or touch a memory pool in the
// middle of a step.  This entry point runs the same planner and chunk kernels
// but keeps the plan in a fixed array that lives in the library's own device
// memory, so it allocates nothing.  It never splits sequences (the split's
// records would not fit a modest fixed array), so each (sequence, head)
// chain runs in one CTA.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace kda {

namespace {

// Fixed scratch: [segment count (int32) | 256-byte pad | Segment[capacity]].
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 256 * 1024;
constexpr size_t kSegOffset = 256;
constexpr int32_t kNoAllocMaxSeqs =
    static_cast<int32_t>((kNoAllocScratchBytes - kSegOffset) / sizeof(Segment));

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the symbol name is only a host-side handle,
// never a device pointer, so kernels always receive this looked-up address.
std::mutex g_mu;
std::vector<unsigned char*> g_addr;

kda_status scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(KDA_ERR_CUDA, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lk(g_mu);
  if (static_cast<int>(g_addr.size()) <= dev) g_addr.resize(dev + 1, nullptr);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[160];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(no-allocation scratch): %s",
               cudaGetErrorString(e));
      return report_error(KDA_ERR_CUDA, msg);
    }
    g_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_addr[dev];
  return KDA_OK;
}

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                            const float* log_alpha, const float* beta,
                                            const float* S0, const int32_t* cu_seqlens,
                                            void* out, float* S_final, int64_t T, int32_t N,
                                            int32_t H, int32_t dk, int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd_noalloc");
  // ---- host-side checks: kda_chunk_fwd's own, plus the scratch limit;
  // nothing is launched on failure
  kda_status st = check_prefill_args(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, T, N,
                                     H, dk, dv, 0, false, 0, nullptr, 0);
  if (st != KDA_OK) return st;
  if (N > kNoAllocMaxSeqs) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "n_seqs=%d exceeds the no-allocation scratch limit of %d sequences; "
             "use kda_chunk_fwd",
             N, kNoAllocMaxSeqs);
    return report_error(KDA_ERR_UNSUPPORTED, msg);
  }
  if (N == 0) return KDA_OK;

  // ---- device work: planner + chunk kernels, plan kept in the fixed scratch
  unsigned char* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  int* err = nullptr;
  st = device_error_word(&err);
  if (st != KDA_OK) return st;

  PrefillArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.log_alpha = log_alpha;
  a.beta = beta;
  a.S0 = S0;
  a.out = static_cast<uint16_t*>(out);
  a.S_final = S_final;
  a.T = T; a.N = N; a.H = H; a.dk = dk; a.dv = dv;
  a.incr_trans = nullptr;   // no split: no increment / transition records
  a.entry_state = nullptr;
  a.plan.n_segs = reinterpret_cast<int32_t*>(scratch);
  a.plan.segs = reinterpret_cast<Segment*>(scratch + kSegOffset);
  a.plan.capacity = N;      // one segment per sequence
  a.err = err;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The planner rewrites the segment count and every segment it emits on each
  // call, so no part of the scratch needs clearing beforehand.
  cudaError_t e = launch_plan(cu_seqlens, T, N, -1, a.plan, err, s);
  if (e == cudaSuccess) e = launch_prefill_replay(a, s);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof msg, "prefill launch: %s", cudaGetErrorString(e));
    return report_error(KDA_ERR_CUDA, msg);
  }
  return KDA_OK;
}
