// kda_chunk_fwd_host: prefill of a uniform batch whose tensors live in host
// memory.  The batch is cut along time into slices of `slice` tokens per
// sequence.  Three streams of the library run the transfers of one slice
// while the kernels of another run: host->device copy of slice i+1 ||
// prefill of slice i || device->host copy of slice i-1.  The state stays on
// the device between slices: each slice starts from the state the previous
// one left (the in-place continuation S_final == S0 that kda_chunk_fwd
// allows), so the result is the single-call result.  Only host code here.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace kda {

namespace {

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t ev[8] = {};  // [0..1] copied in, [2..3] computed, [4..5] copied out, [6] start, [7] spare
};

std::mutex g_pipe_mu;
std::vector<HostPipe> g_pipes;

cudaError_t host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  if ((int)g_pipes.size() <= dev) g_pipes.resize(dev + 1);
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    for (cudaStream_t* s : {&p.in, &p.comp, &p.out}) {
      e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
      if (e != cudaSuccess) return e;
    }
    for (cudaEvent_t& ev : p.ev) {
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_chunk_fwd_host(const void* q, const void* k, const void* v,
                                         const float* log_alpha, const float* beta,
                                         const float* S0, void* out, float* S_final,
                                         int64_t total_tokens, int32_t n_seqs, int32_t H,
                                         int32_t dk, int32_t dv, int64_t slice_tokens,
                                         void* stream_v) {
  NvtxRange nvtx_range("kda_chunk_fwd_host");
  const int64_t T = total_tokens;
  const int32_t N = n_seqs;
  if (T < 0 || N < 0 || H <= 0) return report_error(KDA_ERR_INVALID_ARGUMENT, "bad sizes");
  if (H > kMaxPrefillHeads)
    return report_error(KDA_ERR_UNSUPPORTED, "n_heads exceeds 65535 (the prefill grid's second dimension)");
  if ((dk != 64 && dk != 128) || dv != dk)
    return report_error(KDA_ERR_UNSUPPORTED, "dk == dv in {64, 128} is required");
  if (N == 0 || T == 0) {
    if (N > 0 && T > 0) return report_error(KDA_ERR_INVALID_ARGUMENT, "bad sizes");
    if (N == 0 && T > 0) return report_error(KDA_ERR_INVALID_ARGUMENT, "tokens given but n_seqs = 0");
  }
  if (N > 0 && T % N != 0)
    return report_error(KDA_ERR_INVALID_ARGUMENT, "total_tokens is not a multiple of n_seqs");
  if (slice_tokens < 0 || slice_tokens % kChunk != 0)
    return report_error(KDA_ERR_INVALID_ARGUMENT, "slice_tokens must be 0 or a positive multiple of 64");
  if (T > 0 && (!q || !k || !v || !log_alpha || !beta || !out))
    return report_error(KDA_ERR_INVALID_ARGUMENT, "a required host pointer is NULL");
  if (N == 0) return KDA_OK;

  const int64_t Tb = T / N;  // tokens per sequence
  int64_t L = slice_tokens > 0 ? slice_tokens : 512;
  if (L > Tb) L = Tb;
  const int64_t n_slices = Tb > 0 ? (Tb + L - 1) / L : 0;
  const size_t qk_row = size_t(H) * dk * 2, v_row = size_t(H) * dv * 2;  // bytes per token row
  const size_t la_row = size_t(H) * dk * 4, b_row = size_t(H) * 4;
  const size_t s_bytes = size_t(N) * H * dk * dv * 4;
  const size_t rows = size_t(N) * (L > 0 ? L : 1);  // token rows of one slice

  cudaStream_t s = static_cast<cudaStream_t>(stream_v);
  HostPipe* pp = nullptr;
  cudaError_t e = host_pipe(&pp);
  if (e != cudaSuccess) return report_error(KDA_ERR_CUDA, cudaGetErrorString(e));
  HostPipe& P = *pp;

  // device memory: the state and two sets of slice buffers (each piece 256-byte aligned)
  auto align = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t per_set = 2 * align(rows * qk_row) + 2 * align(rows * v_row) +
                         align(rows * la_row) + align(rows * b_row);
  char* mem = nullptr;
  e = cudaMallocAsync(reinterpret_cast<void**>(&mem), align(s_bytes) + 2 * per_set, s);
  if (e != cudaSuccess) return report_error(KDA_ERR_OUT_OF_MEMORY, cudaGetErrorString(e));
  float* state = reinterpret_cast<float*>(mem);
  struct Set { char *q, *k, *v, *la, *b, *o; } set[2];
  for (int i = 0; i < 2; ++i) {
    char* base = mem + align(s_bytes) + i * per_set;
    set[i].q = base;
    set[i].k = set[i].q + align(rows * qk_row);
    set[i].v = set[i].k + align(rows * qk_row);
    set[i].la = set[i].v + align(rows * v_row);
    set[i].b = set[i].la + align(rows * la_row);
    set[i].o = set[i].b + align(rows * b_row);
  }

  // on a failure, free the memory only after the pipe streams' queued work
  auto release = [&]() {
    for (cudaStream_t t : {P.in, P.comp, P.out})
      if (cudaEventRecord(P.ev[7], t) == cudaSuccess) cudaStreamWaitEvent(s, P.ev[7], 0);
    cudaFreeAsync(mem, s);
  };
  auto fail = [&](cudaError_t err) {
    release();
    return report_error(KDA_ERR_CUDA, cudaGetErrorString(err));
  };
#define KDA_TRY(x) do { cudaError_t _e = (x); if (_e != cudaSuccess) return fail(_e); } while (0)
  // everything below starts after the caller's stream reaches this point
  KDA_TRY(cudaEventRecord(P.ev[6], s));
  for (cudaStream_t t : {P.in, P.comp, P.out}) KDA_TRY(cudaStreamWaitEvent(t, P.ev[6], 0));

  if (S0) KDA_TRY(cudaMemcpyAsync(state, S0, s_bytes, cudaMemcpyHostToDevice, P.in));
  else KDA_TRY(cudaMemsetAsync(state, 0, s_bytes, P.in));

  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  const char* hla = reinterpret_cast<const char*>(log_alpha);
  const char* hb = reinterpret_cast<const char*>(beta);
  char* ho = static_cast<char*>(out);
  kda_status st = KDA_OK;
  // Rows [t0, t0 + len) of every sequence between the host tensor ([N][Tb]
  // rows of rb bytes) and the slice buffer ([N][len] rows): one strided 2-D
  // copy when the host pitch is within the copy engines' limit, else one copy
  // per sequence.
  auto copy_rows = [&](char* dev, const char* host_src, char* host_dst, const char* dev_src,
                       int64_t rb, int64_t t0, int64_t len, cudaMemcpyKind kind,
                       cudaStream_t st_) -> cudaError_t {
    const size_t hp = static_cast<size_t>(Tb * rb), dp = static_cast<size_t>(len * rb);
    if (hp < (size_t(1) << 31)) {
      return kind == cudaMemcpyHostToDevice
                 ? cudaMemcpy2DAsync(dev, dp, host_src + t0 * rb, hp, dp, N, kind, st_)
                 : cudaMemcpy2DAsync(host_dst + t0 * rb, hp, dev_src, dp, dp, N, kind, st_);
    }
    for (int32_t n = 0; n < N; ++n) {
      const int64_t h_row = n * Tb + t0, d_row = n * len;
      const cudaError_t e =
          kind == cudaMemcpyHostToDevice
              ? cudaMemcpyAsync(dev + d_row * rb, host_src + h_row * rb, len * rb, kind, st_)
              : cudaMemcpyAsync(host_dst + h_row * rb, dev_src + d_row * rb, len * rb, kind, st_);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  };
  for (int64_t i = 0; i < n_slices; ++i) {
    const int buf = static_cast<int>(i & 1);
    const int64_t t0 = i * L, len = (Tb - t0) < L ? (Tb - t0) : L;
    Set& B = set[buf];
    // inputs of slice i: the buffers' previous slice (i - 2) must have been computed
    if (i >= 2) KDA_TRY(cudaStreamWaitEvent(P.in, P.ev[2 + buf], 0));
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
    KDA_TRY(copy_rows(B.q, hq, nullptr, nullptr, qk_row, t0, len, h2d, P.in));
    KDA_TRY(copy_rows(B.k, hk, nullptr, nullptr, qk_row, t0, len, h2d, P.in));
    KDA_TRY(copy_rows(B.v, hv, nullptr, nullptr, v_row, t0, len, h2d, P.in));
    KDA_TRY(copy_rows(B.la, hla, nullptr, nullptr, la_row, t0, len, h2d, P.in));
    KDA_TRY(copy_rows(B.b, hb, nullptr, nullptr, b_row, t0, len, h2d, P.in));
    KDA_TRY(cudaEventRecord(P.ev[0 + buf], P.in));
    // prefill of slice i from the device state, in place
    KDA_TRY(cudaStreamWaitEvent(P.comp, P.ev[0 + buf], 0));
    if (i >= 2) KDA_TRY(cudaStreamWaitEvent(P.comp, P.ev[4 + buf], 0));  // out buffer drained
    st = kda_chunk_fwd(B.q, B.k, B.v, reinterpret_cast<const float*>(B.la),
                       reinterpret_cast<const float*>(B.b), state, nullptr, B.o, state,
                       N * len, N, H, dk, dv, P.comp);
    if (st != KDA_OK) { release(); return st; }
    KDA_TRY(cudaEventRecord(P.ev[2 + buf], P.comp));
    // outputs of slice i back to the host
    KDA_TRY(cudaStreamWaitEvent(P.out, P.ev[2 + buf], 0));
    KDA_TRY(copy_rows(nullptr, nullptr, ho, B.o, v_row, t0, len, cudaMemcpyDeviceToHost, P.out));
    KDA_TRY(cudaEventRecord(P.ev[4 + buf], P.out));
  }
  if (S_final) {
    // the last slice's prefill has been waited for by the output stream
    KDA_TRY(cudaStreamWaitEvent(P.out, n_slices > 0 ? P.ev[2 + ((n_slices - 1) & 1)] : P.ev[6], 0));
    KDA_TRY(cudaStreamWaitEvent(P.out, P.ev[6], 0));
    if (n_slices == 0) {  // no tokens: S_final = S0 (or zero)
      KDA_TRY(cudaEventRecord(P.ev[7], P.in));
      KDA_TRY(cudaStreamWaitEvent(P.out, P.ev[7], 0));
    }
    KDA_TRY(cudaMemcpyAsync(S_final, state, s_bytes, cudaMemcpyDeviceToHost, P.out));
  }
  // the caller's stream continues once all three pipe streams are done
  for (cudaStream_t t : {P.in, P.comp, P.out}) {
    KDA_TRY(cudaEventRecord(P.ev[7], t));
    KDA_TRY(cudaStreamWaitEvent(s, P.ev[7], 0));
  }
#undef KDA_TRY
  e = cudaFreeAsync(mem, s);
  if (e != cudaSuccess) return report_error(KDA_ERR_CUDA, cudaGetErrorString(e));
  return KDA_OK;
}
