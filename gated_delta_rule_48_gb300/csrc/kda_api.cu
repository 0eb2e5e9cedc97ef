// Host side of the C ABI (include/kda.h): argument checks, per-device state,
// the stream-ordered workspace, the prefill schedule and launch tracing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace kda {

// Device error word: kernels OR DeviceError flags into it; never trap.
__device__ int g_device_error = 0;

namespace {

thread_local std::string t_last_error;

kda_status fail(kda_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

kda_status cuda_fail(cudaError_t e, const char* what) {
  kda_status st = (e == cudaErrorMemoryAllocation) ? KDA_ERR_OUT_OF_MEMORY : KDA_ERR_CUDA;
  return fail(st, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- per device
// The basic state (SM count, device address of the error word) is set up on
// the first call of any entry point on a device.  The workspace pool is
// created separately, on the first call that needs a workspace, so entry
// points that allocate nothing never create or touch it.
struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int* err = nullptr;          // address of g_device_error on this device
  cudaMemPool_t pool = nullptr;
};

std::mutex g_dev_mu;
std::vector<DeviceState> g_devs;

kda_status device_state(DeviceState** out, bool want_pool = false) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if ((int)g_devs.size() <= dev) g_devs.resize(dev + 1);
  DeviceState& d = g_devs[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
    d.ready = true;
  }
  if (want_pool && !d.pool) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = ~0ull;  // keep freed workspace cached in the pool
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return cuda_fail(e, "cudaMemPoolSetAttribute");
    }
    d.pool = pool;
  }
  *out = &d;
  return KDA_OK;
}

// ---------------------------------------------------------------- tracing
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof_open, g_prof_done;

// ---------------------------------------------------------------- checks
bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

struct Range {
  const char* name;
  uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const char* name, const void* p, int64_t bytes) {
  uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{name, lo, p ? lo + static_cast<uintptr_t>(bytes) : lo};
}

bool overlaps(const Range& a, const Range& b) {
  if (a.lo == a.hi || b.lo == b.hi) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

kda_status check_head_dims(int32_t dk, int32_t dv) {
  if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARGUMENT, "dk=%d dv=%d must be positive", dk, dv);
  if (dk != dv || (dk != 64 && dk != 128))
    return fail(KDA_ERR_UNSUPPORTED, "only dk == dv in {64, 128} is supported (got dk=%d dv=%d)", dk, dv);
  return KDA_OK;
}

}  // namespace

// Error reporting and the device error word for the other translation units.
kda_status report_error(kda_status st, const char* msg) { return fail(st, "%s", msg); }

kda_status device_error_word(int** out) {
  DeviceState* dev = nullptr;
  kda_status st = device_state(&dev);
  if (st == KDA_OK) *out = dev->err;
  return st;
}

void prof_begin(cudaStream_t s, const char* name) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  ProfRecord r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.start) != cudaSuccess) return;
  if (cudaEventCreate(&r.stop) != cudaSuccess) { cudaEventDestroy(r.start); return; }
  cudaEventRecord(r.start, s);
  g_prof_open.push_back(r);
}

void prof_end(cudaStream_t s, const char* name) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  for (size_t i = g_prof_open.size(); i-- > 0;) {
    if (g_prof_open[i].name == name) {
      cudaEventRecord(g_prof_open[i].stop, s);
      g_prof_done.push_back(g_prof_open[i]);
      g_prof_open.erase(g_prof_open.begin() + i);
      return;
    }
  }
}

// Segment length used when the caller asks for the automatic choice.
// Every CTA of the chunk kernels walks one (segment, head) unit at a roughly
// fixed time per 64-token chunk, one CTA per SM, so a pass over U units of at
// most L chunks takes about ceil(U / SMs) waves of L chunk-times.  Unsplit, the
// N H chains take ceil(N H / SMs) waves of the whole sequence.  Split into s
// segments per sequence, a uniform batch's first pass runs N H (s - 1) units
// (the replays of segment 0 and the summaries of segments 1 .. s - 2) and its
// second pass the N H (s - 1) replays of segments 1 .. s - 1; the scan of the
// entry states adds about one chunk-time per segment.  Each wave also pays a fixed start
// (TMEM, the initial state, the first chunk's loads), taken as two
// chunk-times.  The choice is the s with the least modelled time (at least 4
// chunks per segment, at most 8 replay waves), and no split when splitting
// does not beat the unsplit time.
//
// The model takes every sequence as T / N tokens long, which is exact for a
// uniform batch.  A packed batch's lengths live on the device; there the
// first pass only summarises (N H (s - 1) units) and the second replays every
// segment (N H s units), the model counts exactly that, and its shorter
// segments keep both passes balanced when the lengths are very uneven.  (On
// log-uniform length mixes of 1,048,576 tokens, a list-scheduling simulation
// puts that choice within ~3 % of the best fixed length; replaying segment 0
// in the first pass at the uniform count's length lost up to 20 % there.)
static int64_t auto_segment_tokens(int64_t T, int32_t N, int32_t H, int sm_count, bool uniform) {
  if (T <= 0 || N <= 0 || H <= 0 || sm_count <= 0) return -1;
  const int64_t chains = static_cast<int64_t>(N) * H, sms = sm_count;
  if (chains >= sms) return -1;
  const int64_t len = ((T + N - 1) / N + kChunk - 1) / kChunk;  // chunks per sequence
  constexpr int64_t kWaveStart = 2, kMinChunks = 4;
  // A replay that loads its segment's T records from the first pass costs
  // kTinNum / kTinDen of one that computes them; times below are in
  // chunk-times x kTinDen.
  constexpr int64_t kTinNum = 77, kTinDen = 100;
  auto waves = [&](int64_t units) { return (units + sms - 1) / sms; };
  auto cost = [&](int64_t L) {
    const int64_t segs = (len + L - 1) / L, last = len - (segs - 1) * L;
    const int64_t w1 = waves(chains * (segs - 1));
    const int64_t first = w1 * (L + kWaveStart) * kTinDen;
    int64_t second;
    if (uniform) {  // segments 1 .. segs-2 load their records; the last computes its own
      const int64_t longest = std::max(segs > 2 ? kTinNum * L : 0, kTinDen * last);
      second = w1 * (longest + kWaveStart * kTinDen);
    } else {        // lengths unknown here: any segment may be a full-length last one
      second = waves(chains * segs) * (L + kWaveStart) * kTinDen;
    }
    return first + second + segs * kTinDen;
  };
  int64_t best = waves(chains) * (len + kWaveStart) * kTinDen, best_L = -1;
  // beyond 8 waves of replay units every extra segment only adds wave starts
  const int64_t s_max = std::min(len / kMinChunks, std::max<int64_t>(2, 8 * sms / chains));
  for (int64_t s = 2; s <= s_max; ++s) {
    // the lengths that cut a sequence into exactly s segments: (s-1) L < len <= s L
    const int64_t lo = std::max((len + s - 1) / s, kMinChunks);
    const int64_t hi = (len + s - 2) / (s - 1) - 1;
    if (lo > hi) continue;
    // For fixed s the wave counts are fixed, so the modelled time is piecewise
    // linear in L: its minimum is at an end of the range or (uniform) where the
    // loaded segments and the last one take equally long.
    const int64_t bal = len * kTinDen / ((s - 1) * kTinDen + kTinNum);
    const int64_t cand[4] = {lo, hi, bal, bal + 1};
    for (int64_t L : cand) {
      if (L < lo || L > hi) continue;
      const int64_t t = cost(L);
      if (t < best) {
        best = t;
        best_L = L;
      }
    }
  }
  return best_L > 0 ? best_L * kChunk : -1;
}

extern "C" int64_t kda_auto_segment_tokens(int64_t total_tokens, int32_t n_seqs, int32_t n_heads,
                                           int32_t sm_count, int32_t uniform) {
  return auto_segment_tokens(total_tokens, n_seqs, n_heads, sm_count, uniform != 0);
}

// Host-side checks of a prefill call; nothing is launched unless all pass.
// Shared by every prefill entry point that takes device pointers, so they
// reject the same arguments with the same status.
kda_status check_prefill_args(const void* q, const void* k, const void* v,
                              const void* log_alpha, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, const void* out, const float* S_final,
                              int64_t T, int32_t N, int32_t H, int32_t dk, int32_t dv,
                              int64_t segment_tokens, bool fused, int64_t ckpt_interval,
                              const float* ckpt, int64_t ckpt_max) {
  const char* la_name = fused ? "gate" : "log_alpha";
  if (T < 0 || N < 0 || H <= 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "total_tokens=%lld n_seqs=%d n_heads=%d",
                (long long)T, N, H);
  kda_status st = check_head_dims(dk, dv);
  if (st != KDA_OK) return st;
  if (H > kMaxPrefillHeads)  // heads are the second grid dimension of the prefill kernels
    return fail(KDA_ERR_UNSUPPORTED, "n_heads=%d exceeds %d", H, kMaxPrefillHeads);
  if (N == 0 && T > 0) return fail(KDA_ERR_INVALID_ARGUMENT, "tokens given but n_seqs = 0");
  if (!cu_seqlens && N > 0 && T % N != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "cu_seqlens is NULL but total_tokens=%lld is not a multiple of n_seqs=%d",
                (long long)T, N);
  if (segment_tokens > 0 && segment_tokens % kChunk != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "segment_tokens=%lld is not a multiple of %d",
                (long long)segment_tokens, kChunk);
  if (ckpt_interval != 0) {
    if (ckpt_interval < 0 || ckpt_interval % kChunk != 0 || ckpt_interval > 0x7fffffffLL)
      return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoint interval=%lld is not a positive multiple of %d",
                  (long long)ckpt_interval, kChunk);
    if (ckpt_max < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "max_checkpoints=%lld", (long long)ckpt_max);
    if (ckpt_max > 0 && !ckpt) return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoints is NULL");
    if (misaligned(ckpt))
      return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoints is not 16-byte aligned");
  }
  if (T > 0) {
    const struct { const void* p; const char* n; } req[] = {
        {q, "q"}, {k, "k"}, {v, "v"}, {log_alpha, la_name}, {beta, "beta"}, {out, "out"}};
    for (auto& r : req)
      if (!r.p) return fail(KDA_ERR_INVALID_ARGUMENT, "%s is NULL", r.n);
  }
  const void* all[] = {q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final};
  const char* names[] = {"q", "k", "v", la_name, "beta", "S0", "cu_seqlens", "out", "S_final"};
  for (int i = 0; i < 9; ++i)
    if (misaligned(all[i])) return fail(KDA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
  const int64_t qk_bytes = T * H * dk * 2, v_bytes = T * H * dv * 2;
  const int64_t la_bytes = T * H * dk * (fused ? 2 : 4), b_bytes = T * H * 4;
  const int64_t s_bytes = static_cast<int64_t>(N) * H * dk * dv * 4;
  Range in[] = {range_of("q", q, qk_bytes), range_of("k", k, qk_bytes), range_of("v", v, v_bytes),
                range_of(la_name, log_alpha, la_bytes), range_of("beta", beta, b_bytes),
                range_of("S0", S0, S0 ? s_bytes : 0),
                range_of("cu_seqlens", cu_seqlens, cu_seqlens ? (N + 1) * 4 : 0)};
  Range r_out = range_of("out", out, T > 0 ? v_bytes : 0);
  Range r_sf = range_of("S_final", S_final, S_final ? s_bytes : 0);
  const int64_t ck_bytes = (ckpt_interval > 0 && ckpt) ? ckpt_max * H * dk * dv * 4 : 0;
  Range r_ck = range_of("checkpoints", ckpt, ck_bytes);
  for (const Range& r : in)
    if (overlaps(r_ck, r)) return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoints overlap %s", r.name);
  if (overlaps(r_ck, r_out) || overlaps(r_ck, r_sf))
    return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoints overlap out or S_final");
  for (int i = 0; i < 7; ++i) {
    const Range& r = in[i];
    if (overlaps(r_out, r)) return fail(KDA_ERR_INVALID_ARGUMENT, "out overlaps %s", r.name);
    const bool exact_alias = (i == 5) && r.lo == r_sf.lo;  // S_final == S0 is allowed
    if (!exact_alias && overlaps(r_sf, r))
      return fail(KDA_ERR_INVALID_ARGUMENT, "S_final overlaps %s", r.name);
  }
  if (overlaps(r_out, r_sf)) return fail(KDA_ERR_INVALID_ARGUMENT, "out overlaps S_final");
  return KDA_OK;
}


// fused = false: q, k normalised by the caller, log_alpha f32.  fused = true:
// q, k raw, and `log_alpha` points at the bf16 gate logits instead.
static kda_status chunk_fwd_impl(const void* q, const void* k, const void* v,
                                 const void* log_alpha, const float* beta,
                                 const float* S0, const int32_t* cu_seqlens, void* out,
                                 float* S_final, int64_t T, int32_t N, int32_t H,
                                 int32_t dk, int32_t dv, int64_t segment_tokens, bool fused,
                                 int64_t ckpt_interval, float* ckpt, int64_t ckpt_max,
                                 void* stream_v, float* dump = nullptr, int32_t dump_seq = -1,
                                 int32_t dump_head = -1, int64_t dump_chunk = -1) {
  kda_status st = check_prefill_args(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, T,
                                     N, H, dk, dv, segment_tokens, fused, ckpt_interval, ckpt,
                                     ckpt_max);
  if (st != KDA_OK || N == 0) return st;

  // ---- device work
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != KDA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream_v);

  int64_t L = segment_tokens;
  if (L == 0) L = auto_segment_tokens(T, N, H, dev->sm_count, cu_seqlens == nullptr);
  bool split = L > 0 && L < T;
  if (!split) L = -1;
  const int64_t capacity64 = split ? static_cast<int64_t>(N) + (T + L - 1) / L + 1 : N;
  if (capacity64 > (1LL << 30)) return fail(KDA_ERR_UNSUPPORTED, "too many segments");
  if (capacity64 * H > 0x7fffffffLL)  // one block per (segment, head) unit
    return fail(KDA_ERR_UNSUPPORTED, "%lld segments x %d heads exceed the grid",
                (long long)capacity64, H);
  const int32_t capacity = static_cast<int32_t>(capacity64);

  // workspace: [segment count | segments | incr_trans | entry_state |
  //             checkpoint bases | launch orders | T records]
  auto align_up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off_nseg = 0;
  size_t off_segs = align_up(off_nseg + sizeof(int32_t));
  size_t off_it = align_up(off_segs + sizeof(Segment) * capacity);
  // (B | M) records and entry states at the kernels' state width
  size_t it_bytes = split ? sizeof(float) * capacity * H * kStateD * (size_t)(2 * kStateD) : 0;
  size_t off_es = align_up(off_it + it_bytes);
  size_t es_bytes = split ? sizeof(float) * capacity * H * kStateD * (size_t)kStateD : 0;
  const bool want_ckpt = ckpt_interval > 0;  // the planner counts (and flags an overflow) even if max = 0
  size_t off_ck = align_up(off_es + es_bytes);
  size_t ck_base_bytes = want_ckpt ? sizeof(int64_t) * (size_t)N : 0;
  // launch orders, longest segment first: the first pass's, the second pass's, their lengths
  size_t off_ord = align_up(off_ck + ck_base_bytes);
  size_t off_ord2 = align_up(off_ord + sizeof(int32_t) * capacity);
  size_t off_nord = align_up(off_ord2 + sizeof(int32_t) * capacity);
  // T records of the summarised segments (one slot of L / 64 chunks per
  // segment and head), read back by the second pass
  const int64_t t_seg_chunks = split ? L / kChunk : 0;
  size_t off_t = align_up(off_nord + 2 * sizeof(int32_t));
  size_t t_bytes = split ? static_cast<size_t>(capacity) * H * t_seg_chunks * kTChunkBytes : 0;
  size_t ws_bytes = align_up(off_t + t_bytes);

  // A uniform batch with neither split nor checkpoints needs no plan and no
  // workspace: the chunk kernel takes segment i = sequence i.
  const bool direct = !cu_seqlens && !split && !want_ckpt && T > 0;
  char* ws = nullptr;
  cudaError_t e = cudaSuccess;
  if (!direct) {
    st = device_state(&dev, /*want_pool=*/true);
    if (st != KDA_OK) return st;
    // Stream capture turns the allocation into a graph memory node, which takes
    // the default pool; otherwise the library's own pool keeps workspace cached.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    auto alloc = [&](size_t bytes) {
      return cap == cudaStreamCaptureStatusNone
                 ? cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), bytes, dev->pool, s)
                 : cudaMallocAsync(reinterpret_cast<void**>(&ws), bytes, s);
    };
    e = alloc(ws_bytes);
    if (e == cudaErrorMemoryAllocation && t_bytes > 0) {
      // no room for the T records: the second pass recomputes T instead
      (void)cudaGetLastError();
      t_bytes = 0;
      ws_bytes = off_t;
      e = alloc(ws_bytes);
    }
    if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  }

  PrefillArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.log_alpha = fused ? nullptr : static_cast<const float*>(log_alpha);
  a.fused = fused ? 1 : 0;
  a.gate = fused ? static_cast<const uint16_t*>(log_alpha) : nullptr;
  a.beta = beta;
  a.S0 = S0;
  a.out = static_cast<uint16_t*>(out);
  a.S_final = S_final;
  a.T = T; a.N = N; a.H = H; a.dk = dk; a.dv = dv;
  a.incr_trans = split ? reinterpret_cast<float*>(ws + off_it) : nullptr;
  a.entry_state = split ? reinterpret_cast<float*>(ws + off_es) : nullptr;
  a.plan.segs = direct ? nullptr : reinterpret_cast<Segment*>(ws + off_segs);
  a.plan.n_segs = direct ? nullptr : reinterpret_cast<int32_t*>(ws + off_nseg);
  a.plan.capacity = capacity;
  a.plan.order = direct ? nullptr : reinterpret_cast<int32_t*>(ws + off_ord);
  a.plan.order2 = direct ? nullptr : reinterpret_cast<int32_t*>(ws + off_ord2);
  a.plan.n_order = direct ? nullptr : reinterpret_cast<int32_t*>(ws + off_nord);
  a.plan.first_replayed = split && cu_seqlens == nullptr ? 1 : 0;  // uniform batches
  a.t_cache = t_bytes > 0 ? reinterpret_cast<unsigned char*>(ws + off_t) : nullptr;
  a.t_seg_chunks = t_seg_chunks;
  a.plan.t_records = a.t_cache ? 1 : 0;
  if (direct) a.plan.direct_len = T / N;
  if (want_ckpt) {
    a.plan.ckpt_base = reinterpret_cast<int64_t*>(ws + off_ck);
    a.plan.ckpt_interval = ckpt_interval;
    a.plan.ckpt_max = ckpt_max;
    a.ckpt = ckpt_max > 0 ? ckpt : nullptr;
  }
  a.err = dev->err;
  a.dump = dump;  // no split here: segment i is sequence i
  a.dump_seg = dump_seq;
  a.dump_head = dump_head;
  a.dump_chunk = dump_chunk;

  kda_status result = KDA_OK;
  if (!direct) e = launch_plan(cu_seqlens, T, N, L, a.plan, a.err, s);
  if (split) {  // summaries (and, uniform, first segments replayed); scan; replays
    if (e == cudaSuccess) e = launch_prefill_pass1(a, s);
    if (e == cudaSuccess) e = launch_segment_scan(a, s);
    a.pass = 2;
    if (e == cudaSuccess) e = launch_prefill_pass2(a, s);
  } else if (e == cudaSuccess) {
    e = dump ? launch_prefill_replay_dump(a, s) : launch_prefill_replay(a, s);
  }
  if (e != cudaSuccess) result = cuda_fail(e, "prefill launch");
  if (ws) {
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (result == KDA_OK && ef != cudaSuccess) result = cuda_fail(ef, "workspace free");
  }
  return result;
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_chunk_fwd(const void* q, const void* k, const void* v,
                                    const float* log_alpha, const float* beta,
                                    const float* S0, const int32_t* cu_seqlens, void* out,
                                    float* S_final, int64_t total_tokens, int32_t n_seqs,
                                    int32_t n_heads, int32_t dk, int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd");
  return chunk_fwd_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, total_tokens,
                        n_seqs, n_heads, dk, dv, 0, false, 0, nullptr, 0, stream);
}

extern "C" kda_status kda_chunk_fwd_fused(const void* q_raw, const void* k_raw, const void* v,
                                          const void* gate, const float* beta, const float* S0,
                                          const int32_t* cu_seqlens, void* out, float* S_final,
                                          int64_t total_tokens, int32_t n_seqs, int32_t n_heads,
                                          int32_t dk, int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd_fused");
  return chunk_fwd_impl(q_raw, k_raw, v, gate, beta, S0, cu_seqlens, out, S_final, total_tokens,
                        n_seqs, n_heads, dk, dv, 0, true, 0, nullptr, 0, stream);
}

extern "C" kda_status kda_chunk_fwd_split(const void* q, const void* k, const void* v,
                                          const float* log_alpha, const float* beta,
                                          const float* S0, const int32_t* cu_seqlens,
                                          void* out, float* S_final, int64_t total_tokens,
                                          int32_t n_seqs, int32_t n_heads, int32_t dk,
                                          int32_t dv, int64_t segment_tokens, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd_split");
  return chunk_fwd_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, total_tokens,
                        n_seqs, n_heads, dk, dv, segment_tokens, false, 0, nullptr, 0,
                        stream);
}

extern "C" kda_status kda_chunk_fwd_checkpoints(const void* q, const void* k, const void* v,
                                                const float* log_alpha, const float* beta,
                                                const float* S0, const int32_t* cu_seqlens,
                                                void* out, float* S_final, int64_t total_tokens,
                                                int32_t n_seqs, int32_t n_heads, int32_t dk,
                                                int32_t dv, int64_t interval, float* checkpoints,
                                                int64_t max_checkpoints, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd_checkpoints");
  if (interval <= 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoint interval=%lld is not a positive multiple of %d",
                (long long)interval, kChunk);
  return chunk_fwd_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, total_tokens,
                        n_seqs, n_heads, dk, dv, 0, false, interval, checkpoints, max_checkpoints,
                        stream);
}

extern "C" kda_status kda_debug_chunk_dump(const void* q, const void* k, const void* v,
                                           const float* log_alpha, const float* beta,
                                           const float* S0, const int32_t* cu_seqlens, void* out,
                                           float* S_final, int64_t total_tokens, int32_t n_seqs,
                                           int32_t n_heads, int32_t dk, int32_t dv, int32_t seq,
                                           int32_t head, int64_t chunk, float* dump,
                                           void* stream) {
  NvtxRange nvtx_range("kda_debug_chunk_dump");
  if (!dump) return fail(KDA_ERR_INVALID_ARGUMENT, "dump is NULL");
  if (misaligned(dump)) return fail(KDA_ERR_INVALID_ARGUMENT, "dump is not 16-byte aligned");
  if (seq < 0 || seq >= n_seqs || head < 0 || head >= n_heads || chunk < 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "seq=%d head=%d chunk=%lld out of range", seq, head,
                (long long)chunk);
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dump),
                  d1 = d0 + static_cast<uintptr_t>(kDumpFloats) * sizeof(float);
  const struct { const void* p; int64_t n; } others[] = {
      {q, total_tokens * n_heads * dk * 2}, {k, total_tokens * n_heads * dk * 2},
      {v, total_tokens * n_heads * dv * 2}, {log_alpha, total_tokens * n_heads * dk * 4},
      {beta, total_tokens * n_heads * 4}, {out, total_tokens * n_heads * dv * 2},
      {S0, S0 ? static_cast<int64_t>(n_seqs) * n_heads * dk * dv * 4 : 0},
      {S_final, S_final ? static_cast<int64_t>(n_seqs) * n_heads * dk * dv * 4 : 0},
      {cu_seqlens, cu_seqlens ? (static_cast<int64_t>(n_seqs) + 1) * 4 : 0}};
  for (const auto& o : others) {
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(o.p), b1 = b0 + static_cast<uintptr_t>(o.n);
    if (o.p && o.n > 0 && d0 < b1 && b0 < d1)
      return fail(KDA_ERR_INVALID_ARGUMENT, "dump overlaps another argument");
  }
  return chunk_fwd_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final, total_tokens,
                        n_seqs, n_heads, dk, dv, -1, false, 0, nullptr, 0, stream, dump, seq,
                        head, chunk);
}

// fused as in chunk_fwd_impl.  K tokens per sequence; commit: device [N] or null.
static kda_status decode_impl(const void* q, const void* k, const void* v, const void* log_alpha,
                              const float* beta, float* S_inout, void* out, const int32_t* commit,
                              int32_t N, int32_t K, int32_t H, int32_t dk, int32_t dv, bool fused,
                              void* stream) {
  const char* la_name = fused ? "gate" : "log_alpha";
  if (N < 0 || H <= 0 || K <= 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "n_seqs=%d n_tokens=%d n_heads=%d", N, K, H);
  kda_status st = check_head_dims(dk, dv);
  if (st != KDA_OK) return st;
  if (N == 0) return KDA_OK;
  const struct { const void* p; const char* n; } req[] = {
      {q, "q"}, {k, "k"}, {v, "v"}, {log_alpha, la_name},
      {beta, "beta"}, {S_inout, "S_inout"}, {out, "out"}};
  for (auto& r : req) {
    if (!r.p) return fail(KDA_ERR_INVALID_ARGUMENT, "%s is NULL", r.n);
    if (misaligned(r.p)) return fail(KDA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", r.n);
  }
  if (misaligned(commit)) return fail(KDA_ERR_INVALID_ARGUMENT, "commit is not 16-byte aligned");
  const int64_t nh = static_cast<int64_t>(N) * H;
  const int64_t th = nh * K;  // (token, head) rows
  Range r_out = range_of("out", out, th * dv * 2);
  Range others[] = {range_of("q", q, th * dk * 2), range_of("k", k, th * dk * 2),
                    range_of("v", v, th * dv * 2),
                    range_of(la_name, log_alpha, th * dk * (fused ? 2 : 4)),
                    range_of("beta", beta, th * 4),
                    range_of("commit", commit, commit ? static_cast<int64_t>(N) * 4 : 0),
                    range_of("S_inout", S_inout, nh * dk * dv * 4)};
  for (auto& r : others)
    if (overlaps(r_out, r)) return fail(KDA_ERR_INVALID_ARGUMENT, "out overlaps %s", r.name);
  for (int i = 0; i < 6; ++i)
    if (overlaps(others[6], others[i]))
      return fail(KDA_ERR_INVALID_ARGUMENT, "S_inout overlaps %s", others[i].name);
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != KDA_OK) return st;
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.log_alpha = fused ? nullptr : static_cast<const float*>(log_alpha);
  a.gate = fused ? static_cast<const uint16_t*>(log_alpha) : nullptr;
  a.beta = beta;
  a.S = S_inout;
  a.out = static_cast<uint16_t*>(out);
  a.commit = commit;
  a.N = N; a.K = K; a.H = H; a.dk = dk; a.dv = dv;
  a.err = dev->err;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KDA_OK;
}

extern "C" kda_status kda_decode_step(const void* q, const void* k, const void* v,
                                      const float* log_alpha, const float* beta,
                                      float* S_inout, void* out, int32_t N, int32_t H,
                                      int32_t dk, int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_decode_step");
  return decode_impl(q, k, v, log_alpha, beta, S_inout, out, nullptr, N, 1, H, dk, dv, false,
                     stream);
}

extern "C" kda_status kda_decode_step_fused(const void* q_raw, const void* k_raw, const void* v,
                                            const void* gate, const float* beta, float* S_inout,
                                            void* out, int32_t N, int32_t H, int32_t dk,
                                            int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_decode_step_fused");
  return decode_impl(q_raw, k_raw, v, gate, beta, S_inout, out, nullptr, N, 1, H, dk, dv, true,
                     stream);
}

extern "C" kda_status kda_decode_tokens_fused(const void* q_raw, const void* k_raw,
                                              const void* v, const void* gate,
                                              const float* beta, float* S_inout, void* out,
                                              const int32_t* commit, int32_t N, int32_t K,
                                              int32_t H, int32_t dk, int32_t dv, void* stream) {
  NvtxRange nvtx_range("kda_decode_tokens_fused");
  return decode_impl(q_raw, k_raw, v, gate, beta, S_inout, out, commit, N, K, H, dk, dv, true,
                     stream);
}

extern "C" kda_status kda_decode_tokens(const void* q, const void* k, const void* v,
                                        const float* log_alpha, const float* beta,
                                        float* S_inout, void* out, const int32_t* commit,
                                        int32_t N, int32_t K, int32_t H, int32_t dk, int32_t dv,
                                        void* stream) {
  NvtxRange nvtx_range("kda_decode_tokens");
  return decode_impl(q, k, v, log_alpha, beta, S_inout, out, commit, N, K, H, dk, dv, false,
                     stream);
}

extern "C" kda_status kda_get_device_error(void* stream) {
  NvtxRange nvtx_range("kda_get_device_error");
  DeviceState* dev = nullptr;
  kda_status st = device_state(&dev);
  if (st != KDA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, dev->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word == 0) return KDA_OK;
  int zero = 0;
  e = cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  std::string msg;
  if (word & kDevErrCuSeqlens)
    msg += "cu_seqlens is malformed (cu[0] != 0, decreasing, or cu[N] != total_tokens); ";
  if (word & kDevErrCapacity) msg += "segment plan exceeded its workspace; ";
  if (word & kDevErrTimeout)
    msg += "a kernel timed out waiting for its asynchronous copies or tensor-core work; ";
  if (word & kDevErrCommit) msg += "a decode commit count is outside [0, n_tokens]; ";
  if (word & kDevErrCheckpoints)
    msg += "the sequences have more checkpoints than max_checkpoints (the excess was dropped); ";
  if (word & kDevErrBounds)
    msg += "a kernel index fell outside its buffer (bounds-checked build; the access was skipped); ";
  return fail(KDA_ERR_DEVICE_INPUT, "%s", msg.c_str());
}

extern "C" kda_status kda_selftest_bounded_wait(uint32_t polls, void* stream) {
  NvtxRange nvtx_range("kda_selftest_bounded_wait");
  if (polls == 0 || polls > (1u << 20))
    return fail(KDA_ERR_INVALID_ARGUMENT, "polls must be in [1, 2^20] (got %u)", polls);
  DeviceState* dev = nullptr;
  kda_status st = device_state(&dev);
  if (st != KDA_OK) return st;
  const cudaError_t e =
      launch_bounded_wait_selftest(polls, dev->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return KDA_OK;
}

extern "C" kda_status kda_selftest_bounds_check(void* stream) {
  NvtxRange nvtx_range("kda_selftest_bounds_check");
  DeviceState* dev = nullptr;
  kda_status st = device_state(&dev);
  if (st != KDA_OK) return st;
  const cudaError_t e = launch_bounds_guard_selftest(dev->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return KDA_OK;
}

extern "C" int kda_bounds_checked(void) { return kBoundsChecked ? 1 : 0; }

extern "C" int64_t kda_workspace_pool_bytes(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev < (int)g_devs.size()) pool = g_devs[dev].pool;
  }
  if (!pool) return -1;
  uint64_t reserved = 0;
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &reserved) != cudaSuccess)
    return -1;
  return static_cast<int64_t>(reserved);
}

extern "C" const char* kda_status_string(kda_status status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_OUT_OF_MEMORY: return "KDA_ERR_OUT_OF_MEMORY";
    case KDA_ERR_DEVICE_INPUT: return "KDA_ERR_DEVICE_INPUT";
  }
  return "unknown kda_status";
}

extern "C" const char* kda_last_error_message(void) { return t_last_error.c_str(); }

extern "C" int kda_abi_version(void) { return KDA_ABI_VERSION; }

extern "C" void kda_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
}

extern "C" int kda_profile_read(kda_kernel_time* entries, int max_entries) {
  cudaDeviceSynchronize();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  std::vector<kda_kernel_time> acc;
  for (auto& r : g_prof_done) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.start, r.stop);
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
    auto it = std::find_if(acc.begin(), acc.end(),
                           [&](const kda_kernel_time& t) { return strcmp(t.name, r.name) == 0; });
    if (it == acc.end()) {
      kda_kernel_time t;
      memset(&t, 0, sizeof t);
      strncpy(t.name, r.name, sizeof(t.name) - 1);
      acc.push_back(t);
      it = acc.end() - 1;
    }
    it->launches += 1;
    it->total_ms += ms;
  }
  g_prof_done.clear();
  int n = 0;
  for (auto& t : acc) {
    if (n >= max_entries || !entries) break;
    entries[n++] = t;
  }
  return n;
}
