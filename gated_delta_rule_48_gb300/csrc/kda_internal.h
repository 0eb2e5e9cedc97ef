// Internal declarations shared by the library's translation units.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;      // tokens per chunk
constexpr int kStateD = 128;    // width of the chunk kernels' states: d = 64 runs
                                // zero-padded to 128 (exact: see kda_prefill_tc.cu)
// The prefill kernels put heads on the grid's second dimension.
constexpr int kMaxPrefillHeads = 65535;
constexpr int kSubTile = 16;    // tokens per decay tile inside a chunk
constexpr float kLogAlphaMin = -5.0f;

// Device error codes (bit flags OR-ed into the device error word).
enum DeviceError : int {
  kDevErrNone = 0,
  kDevErrCuSeqlens = 1,      // cu_seqlens malformed
  kDevErrCapacity = 2,       // more segments than the workspace holds
  kDevErrTimeout = 4,        // a kernel gave up waiting on its own async copies / MMAs
  kDevErrCommit = 8,         // a decode commit count outside [0, tokens per call]
  kDevErrCheckpoints = 16,   // more prefill checkpoints than the caller's buffer holds
  kDevErrBounds = 32,        // bounds-checked build: an index fell outside its buffer
};

// ---- bounds-checked build.  Compiled with -DKDA_BOUNDS_CHECK, every plain
// global-memory access of the kernels (the TMA copies check their own boxes
// against the tensor maps) first asks kda_guard whether elements
// [i, i + width) lie inside a buffer of n elements.  Out of range, the access
// is skipped and kDevErrBounds is set in the device error word: the kernel
// never traps and never touches memory it does not own.  Without the flag the
// guard is the constant true and the checks compile away.
#ifdef KDA_BOUNDS_CHECK
constexpr bool kBoundsChecked = true;
__device__ __forceinline__ bool kda_guard(int64_t i, int64_t width, int64_t n, int* err) {
  if (i >= 0 && width >= 0 && i + width <= n) return true;
  atomicOr(err, kDevErrBounds);
  return false;
}
#else
constexpr bool kBoundsChecked = false;
__device__ __forceinline__ constexpr bool kda_guard(int64_t, int64_t, int64_t, int*) {
  return true;
}
#endif

// One segment of one sequence: tokens [t0, t1) (global indices).
struct Segment {
  int64_t t0, t1;
  int32_t seq;     // sequence index
  int32_t index;   // segment index within its sequence
  int32_t count;   // number of segments of that sequence
  int32_t first;   // global id of that sequence's first segment
};

// Output of the planner, in device memory.
struct Plan {
  Segment* segs;       // [capacity]
  int32_t* n_segs;     // [1] number of valid segments
  int32_t capacity;
  // prefill state checkpoints (ckpt_interval > 0): sequence n's checkpoint j
  // (the state after its first j * ckpt_interval tokens, j >= 1) goes to slot
  // ckpt_base[n] + j - 1 of the caller's buffer, slots >= ckpt_max dropped
  int64_t* ckpt_base = nullptr;  // [N], written by the planner
  int64_t ckpt_interval = 0;
  int64_t ckpt_max = 0;
  // > 0: a uniform batch with neither split nor checkpoints, launched without
  // the planner -- segment i is sequence i, direct_len tokens long
  int64_t direct_len = 0;
  // Launch orders written by the planner, each longest first (decreasing
  // modelled time: the chunk count, scaled for replays that load T records):
  // order [capacity] for the first pass, order2 [capacity] for
  // the second pass of a split prefill, n_order [2] their lengths; order null:
  // rank = segment id.  Unsplit: order lists every segment.  Split with
  // first_replayed: order = every segment but the last one of a split
  // sequence, order2 = the segments with index >= 1.  Split otherwise: order =
  // every segment but the last one of its sequence, order2 = every segment.
  // (A sequence shorter than the segment length is one segment, its last.)
  int32_t* order = nullptr;
  int32_t* order2 = nullptr;
  int32_t* n_order = nullptr;
  // split prefills: 1 when the first pass replays segment 0 of every sequence
  // (uniform batches), 0 when it only summarises (every segment but the last)
  // and the second pass replays all segments (packed batches)
  int32_t first_replayed = 0;
  // the first pass keeps T records for the second (PrefillArgs::t_cache): the
  // second pass's launch order then counts a summarised segment's chunks at
  // 0.77 chunk-times each
  int32_t t_records = 0;
};

// Problem description shared by the prefill kernels.
struct PrefillArgs {
  const uint16_t* q;       // bf16 [T, H, dk]
  const uint16_t* k;
  const uint16_t* v;       // bf16 [T, H, dv]
  const float* log_alpha;  // f32 [T, H, dk]
  const float* beta;       // f32 [T, H]
  const float* S0;         // f32 [N, H, dk, dv] or null
  uint16_t* out;           // bf16 [T, H, dv]
  float* S_final;          // f32 [N, H, dk, dv] or null
  int64_t T;
  int32_t N, H, dk, dv;
  // split workspace (null when sequences are not split)
  float* incr_trans;       // [capacity, H, dk, dv + dk]: B_j | M_j of each segment
  float* entry_state;      // [capacity, H, dk, dv]: S_in(j) for j >= 1
  Plan plan;               // segment list in the workspace
  int* err;                // device error word
  // fused input preparation (kda_chunk_fwd_fused): q, k are raw and are
  // L2-normalised on load; log alpha comes from the bf16 gate logits
  int fused = 0;
  const uint16_t* gate = nullptr;  // bf16 [T, H, dk] when fused
  float* ckpt = nullptr;           // f32 [ckpt_max, H, dk, dv] state checkpoints, or null
  // intermediate dump (kda_debug_chunk_dump): the replay of segment dump_seg,
  // head dump_head writes chunk dump_chunk's intermediates to dump (layout:
  // the kDump* offsets below), or null
  float* dump = nullptr;
  int32_t dump_seg = -1, dump_head = -1;
  int64_t dump_chunk = -1;
  int pass = 1;  // which launch order the kernels walk (2: a split prefill's second pass)
  // Split prefill: the first pass's summaries store each chunk's T (its tf32
  // copy, then the bf16 hi and lo halves: kTChunkBytes) at
  // ((segment * H + head) * t_seg_chunks + chunk) * kTChunkBytes, and the
  // second pass's replays of those segments load it instead of recomputing
  // it.  Null: every replay computes its own T.
  unsigned char* t_cache = nullptr;
  int64_t t_seg_chunks = 0;  // chunks per segment slot (the split's segment length)
};

constexpr int64_t kTChunkBytes = 32768;

// Layout of the intermediate dump, in floats: g [64][128], A_kk [64][64],
// A_qk [64][64], T [64][64], U [64][128], S at the chunk's start [128][128]
// (row = key channel).
constexpr int64_t kDumpG = 0, kDumpAkk = 64 * 128, kDumpAqk = kDumpAkk + 64 * 64,
                  kDumpT = kDumpAqk + 64 * 64, kDumpU = kDumpT + 64 * 64,
                  kDumpS = kDumpU + 64 * 128, kDumpFloats = kDumpS + 128 * 128;

// ---- error reporting shared by the entry points (kda_api.cu)
kda_status report_error(kda_status st, const char* msg);  // sets kda_last_error_message()
kda_status device_error_word(int** out);                   // current device's error word
// Host-side checks shared by the prefill entry points that take device
// pointers (kda_api.cu); KDA_OK when the call may go ahead.
kda_status check_prefill_args(const void* q, const void* k, const void* v,
                              const void* log_alpha, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, const void* out, const float* S_final,
                              int64_t T, int32_t N, int32_t H, int32_t dk, int32_t dv,
                              int64_t segment_tokens, bool fused, int64_t ckpt_interval,
                              const float* ckpt, int64_t ckpt_max);

// ---- tracing: every C entry point opens an NVTX range named after itself
// for its host-side duration (validation, planning, launches), so profilers
// that record NVTX (Nsight Systems, ncu --nvtx) attribute the library's
// kernels to the call that issued them.  Without such a tool attached the
// push and pop are no-ops.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---- launch-time tracing (kda_api.cu)
void prof_begin(cudaStream_t s, const char* name);
void prof_end(cudaStream_t s, const char* name);

// ---- planner and scan (kda_plan.cu)
cudaError_t launch_plan(const int32_t* cu_seqlens, int64_t T, int32_t N,
                        int64_t segment_tokens, Plan plan, int* err,
                        cudaStream_t s);
cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s);

// ---- chunked prefill (kda_prefill_*.cu)
// tcgen05 kernels (kda_prefill_tc.cu), dk = dv = 128 or 64.  Split prefill:
// pass 1 summarises (B_j, M_j) every segment but the last of its sequence,
// except that uniform batches (plan.first_replayed) replay the first segment
// from S0 instead, in the same launch; the scan chains the entry states;
// pass 2 (a.pass = 2) replays the rest, loading the T records of the
// summarised segments.  Unsplit: one replay.
cudaError_t launch_prefill_pass1(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_prefill_pass2(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_prefill_replay(const PrefillArgs& a, cudaStream_t s);
// the replay with the intermediate dump of a.dump (one chunk of one unit)
cudaError_t launch_prefill_replay_dump(const PrefillArgs& a, cudaStream_t s);

// ---- decode (kda_decode.cu)
struct DecodeArgs {
  const uint16_t* q;        // bf16 [N*K, H, dk]
  const uint16_t* k;
  const uint16_t* v;        // bf16 [N*K, H, dv]
  const float* log_alpha;   // f32 [N*K, H, dk]; null when gate is given
  const uint16_t* gate;     // bf16 [N*K, H, dk] logits (fused preparation) or null
  const float* beta;        // f32 [N*K, H]
  float* S;                 // f32 [N, H, dk, dv], updated in place
  uint16_t* out;            // bf16 [N*K, H, dv]
  const int32_t* commit;    // [N] tokens to commit per sequence, or null (all K)
  int32_t N, K, H, dk, dv;
  int* err;                 // device error word
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// K > 1 tokens per sequence (kda_decode_tokens.cu); launch_decode dispatches to it
cudaError_t launch_decode_tokens(const DecodeArgs& a, cudaStream_t s);
// kda_selftest.cu: a bounded wait on an mbarrier nothing arrives on
cudaError_t launch_bounded_wait_selftest(uint32_t polls, int* err, cudaStream_t s);
// kda_selftest.cu: one out-of-range bounds guard (records kDevErrBounds only in
// the bounds-checked build; accesses no memory in either build)
cudaError_t launch_bounds_guard_selftest(int* err, cudaStream_t s);

// bf16 helpers usable from device code without cuda_bf16.h conversions.
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// round to nearest even; NaN stays NaN
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0;
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ float clamp_log_alpha(float la) {
  return fminf(fmaxf(la, kLogAlphaMin), 0.0f);
}

// ---- fused input preparation (the *_fused entry points)
// log alpha from a gate logit x: the bounded gate -5 sigmoid(x), then the
// same clamp as a given log alpha (a no-op for finite x).
__device__ __forceinline__ float gate_log_alpha(float x) {
  return clamp_log_alpha(-5.0f * __frcp_rn(1.0f + __expf(-x)));
}
// Scale of an L2 normalisation x / max(||x||, 1e-12) from ss = sum of x^2.
__device__ __forceinline__ float l2_scale(float ss) {
  return fminf(__frsqrt_rn(ss), 1e12f);
}

}  // namespace kda
