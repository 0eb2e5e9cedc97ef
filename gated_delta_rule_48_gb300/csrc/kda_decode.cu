// Single-token recurrent decode step, state updated in place.
//
// Per (sequence, head), with S of shape D x D (fp32, row c = key channel):
//   S' = Diag(alpha) S,  a = S'^T k,  b = S'^T q,  u = beta (v - a),
//   S  = S' + k u^T  (written back),  o = S^T q = b + (q . k) u.
// One token costs one read and one write of the state, whatever the context
// length (lecture "Inside Kimi K3: Architecture of an Open Frontier Model",
// sequence paragraph: constant cost per new token; orkas.ai close read,
// section "The bill comes due in the serving stack": the state is updated in
// place).
//
// Memory-bound: 8 D^2 bytes of state traffic per (sequence, head) against
// ~7 D^2 flops.  One CTA per (sequence, head); each thread keeps D/8 rows x 4
// columns of the state in registers, loaded with 128-bit streaming loads
// issued before any other work, so the whole 64 KiB tile is in flight at once.
// A warp reads whole 512-byte rows (D = 128), so every access is coalesced.
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

namespace {

template <int D>
struct DecodeCfg {
  static constexpr int kColGroups = D / 4;                 // float4 columns
  static constexpr int kThreads = D == 128 ? 256 : 128;
  static constexpr int kRowGroups = kThreads / kColGroups;  // 8
  static constexpr int kRowsPerThread = D / kRowGroups;     // 16 or 8
};

// K tokens per sequence, applied in order from the state in registers.
// launch_decode runs it for K = 1, the plain step; calls with K > 1 go to the
// persistent multi-token kernel (kda_decode_tokens.cu), which computes the
// same recurrence faster at K > 1.  Token t of sequence n is row n*K + t of the packed
// inputs: q, k, log_alpha [N*K, H, dk], v [N*K, H, dv], beta [N*K, H], out
// [N*K, H, dv].  Every token's output is written; the state in memory
// advances by the first `commit[n]` tokens only (commit == null: all K),
// written back once -- the speculative-decoding form, where a verify call
// commits nothing and a second call over the cached inputs commits the
// accepted prefix (orkas.ai close read, section "The bill comes due in the
// serving stack": an in-place update cannot be undone, so the state is
// rebuilt from the accepted inputs instead of rolled back).
// FUSED: q, k arrive raw and are L2-normalised (then rounded to bf16) here,
// and `gate` (bf16 logits) replaces log_alpha: log alpha = -5 sigmoid(gate).
template <int D, bool FUSED>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads)
decode_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
              const uint16_t* __restrict__ v, const float* __restrict__ log_alpha,
              const uint16_t* __restrict__ gate, const float* __restrict__ beta,
              float* __restrict__ S, uint16_t* __restrict__ out,
              const int32_t* __restrict__ commit, int32_t K, int32_t H, int* __restrict__ err) {
  using Cfg = DecodeCfg<D>;
  constexpr int CG = Cfg::kColGroups, RG = Cfg::kRowGroups, RPT = Cfg::kRowsPerThread;
  const int64_t unit = blockIdx.x;  // sequence * H + head
  const int64_t n = unit / H, h = unit % H;
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;
  // extents (bounds-checked build): units = N H, tokens = N K
  const int64_t units = gridDim.x, n_tok_h = units * K;

  int n_commit = K;
  if (commit) {
    if (!kda_guard(n, 1, units / H, err)) return;
    n_commit = commit[n];
    if (n_commit < 0 || n_commit > K) {  // rejected: nothing is written for this unit
      if (tid == 0) atomicOr(err, kDevErrCommit);
      return;
    }
  }

  __shared__ float s_k[D], s_q[D], s_alpha[D], s_u[D];
  __shared__ __align__(16) float s_red_a[RG][D + 4];
  __shared__ __align__(16) float s_red_b[RG][D + 4];
  __shared__ float s_qk;
  __shared__ float s_scale[2];

  // state tile: rows rg*RPT .. rg*RPT+RPT-1, columns 4*cg .. 4*cg+3
  float4* Sp = reinterpret_cast<float4*>(S + unit * D * D);
  float4 st[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    st[i] = kda_guard(unit * D * D + 4 * ((rg * RPT + i) * CG + cg), 4, units * D * D, err)
                ? __ldcs(&Sp[(rg * RPT + i) * CG + cg])
                : make_float4(0.f, 0.f, 0.f, 0.f);

  // Token t's vectors are loaded into registers (thread c < D: channel c)
  // while token t-1 is computed, so their latency is hidden after the first.
  static_assert(Cfg::kThreads >= D, "one thread per channel");
  const bool chan = tid < D;
  uint16_t pk = 0, pq = 0, pv = 0, pg = 0;
  float pla = 0.f, pb = 0.f;
  auto fetch = [&](int t) {
    const int64_t row = (n * K + t) * H + h;
    if (chan && kda_guard(row * D + tid, 1, n_tok_h * D, err)) {
      const int64_t e = row * D + tid;
      pk = k[e];
      pq = q[e];
      pv = v[e];
      if (FUSED) pg = gate[e]; else pla = log_alpha[e];
    }
    if (kda_guard(row, 1, n_tok_h, err)) pb = beta[row];
  };
  fetch(0);

  for (int t = 0; t < K; ++t) {
    const int64_t row = (n * K + t) * H + h;  // packed (token, head) row
    const int64_t vec = row * D;
    const float vt = bf16_to_f32(pv), bt = pb;
    if (chan) {
      s_k[tid] = bf16_to_f32(pk);
      s_q[tid] = bf16_to_f32(pq);
      s_alpha[tid] = expf(FUSED ? gate_log_alpha(bf16_to_f32(pg)) : clamp_log_alpha(pla));
    }
    if (t + 1 < K) fetch(t + 1);
    __syncthreads();
    if (FUSED) {  // warp 0 normalises k, warp 1 q
      if (tid < 64) {
        const float* x = tid < 32 ? s_k : s_q;
        float ss = 0.f;
        for (int c = tid & 31; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((tid & 31) == 0) s_scale[tid >> 5] = l2_scale(ss);
      }
      __syncthreads();
      for (int c = tid; c < D; c += Cfg::kThreads) {
        s_k[c] = bf16_to_f32(f32_to_bf16(s_k[c] * s_scale[0]));
        s_q[c] = bf16_to_f32(f32_to_bf16(s_q[c] * s_scale[1]));
      }
      __syncthreads();
    }

    if (tid < 32) {  // q . k
      float p = 0.f;
      for (int c = tid; c < D; c += 32) p += s_q[c] * s_k[c];
#pragma unroll
      for (int o = 16; o; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      if (tid == 0) s_qk = p;
    }

    float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg * RPT + i;
      const float al = s_alpha[r], kr = s_k[r], qr = s_q[r];
      st[i].x *= al; st[i].y *= al; st[i].z *= al; st[i].w *= al;
      a[0] += st[i].x * kr; a[1] += st[i].y * kr; a[2] += st[i].z * kr; a[3] += st[i].w * kr;
      b[0] += st[i].x * qr; b[1] += st[i].y * qr; b[2] += st[i].z * qr; b[3] += st[i].w * qr;
    }
    *reinterpret_cast<float4*>(&s_red_a[rg][4 * cg]) = make_float4(a[0], a[1], a[2], a[3]);
    *reinterpret_cast<float4*>(&s_red_b[rg][4 * cg]) = make_float4(b[0], b[1], b[2], b[3]);
    __syncthreads();

    if (chan) {  // column = this thread's channel
      const int col = tid;
      float sa = 0.f, sb = 0.f;
#pragma unroll
      for (int r = 0; r < RG; ++r) { sa += s_red_a[r][col]; sb += s_red_b[r][col]; }
      const float u = bt * (vt - sa);
      s_u[col] = u;
      if (kda_guard(vec + col, 1, n_tok_h * D, err)) out[vec + col] = f32_to_bf16(sb + s_qk * u);
    }
    __syncthreads();

    const float u0 = s_u[4 * cg], u1 = s_u[4 * cg + 1], u2 = s_u[4 * cg + 2], u3 = s_u[4 * cg + 3];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float kr = s_k[rg * RPT + i];
      st[i].x += kr * u0; st[i].y += kr * u1; st[i].z += kr * u2; st[i].w += kr * u3;
    }
    if (t + 1 == n_commit) {
#pragma unroll
      for (int i = 0; i < RPT; ++i)
        if (kda_guard(unit * D * D + 4 * ((rg * RPT + i) * CG + cg), 4, units * D * D, err))
          __stcs(&Sp[(rg * RPT + i) * CG + cg], st[i]);
    }
    if (t + 1 < K) __syncthreads();  // s_k, s_q, s_u are rewritten by the next token
  }
}

template <int D, bool FUSED>
void launch_decode_t(const DecodeArgs& a, int64_t units, cudaStream_t s) {
  decode_kernel<D, FUSED><<<static_cast<unsigned>(units), DecodeCfg<D>::kThreads, 0, s>>>(
      a.q, a.k, a.v, a.log_alpha, a.gate, a.beta, a.S, a.out, a.commit, a.K, a.H, a.err);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.K > 1) return launch_decode_tokens(a, s);  // several tokens: the column-owner kernel
  const int64_t units = static_cast<int64_t>(a.N) * a.H;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prof_begin(s, "kda_decode_step");
  const bool fused = a.gate != nullptr;
  if (a.dk == 128) {
    if (fused) launch_decode_t<128, true>(a, units, s);
    else launch_decode_t<128, false>(a, units, s);
  } else {
    if (fused) launch_decode_t<64, true>(a, units, s);
    else launch_decode_t<64, false>(a, units, s);
  }
  prof_end(s, "kda_decode_step");
  return cudaGetLastError();
}

}  // namespace kda
