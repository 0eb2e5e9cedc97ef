// Multi-token recurrent decode: K tokens per sequence in one call, the state
// kept in registers across them.
//
// Per (sequence, head) and token, with S of shape D x D (fp32, row i = key
// channel, column j = value channel):
//   S' = Diag(alpha) S,  a = S'^T k,  u = beta (v - a),
//   S  = S' + k u^T,     o = S^T q = S'^T q + (q . k) u.
// Inside a batch of 8 tokens the registers hold Z = Diag(P)^{-1} S, with P_t
// the running product of alpha over the batch's tokens 1..t (per key
// channel): then a = (k P)^T Z, S'^T q = (q P)^T Z and Z += (k / P) u^T, three
// multiply-adds per state element and token instead of four.  Z is scaled back
// (S = P Z) where the state is stored and at the end of every batch.  P >=
// e^{-40} within a batch (log alpha >= -5), so Z stays far inside the f32 range
// for any state below ~1e21 in magnitude.
// The inputs and the commit rule are those of the single step (every token's
// output is written; the state in memory advances by the first commit[n]
// tokens, written back once: the speculative-decoding verify / commit form of
// the orkas.ai close read, section "The bill comes due in the serving stack").
//
// Persistent: two (D = 128) or four (D = 64) CTAs of 2D threads per SM, each
// walking (sequence, head) units with a stride of the grid.  While a unit is
// computed from registers, the next unit's state (64 KiB at D = 128) streams
// into shared memory by one bulk asynchronous copy, so its HBM read overlaps
// the arithmetic; the committed state goes from registers straight to HBM.
//
// Thread (p, quarter) owns the state columns j = 2p, 2p + 1 over rows
// [quarter D/4, quarter D/4 + D/4).  A warp holds one quarter (D/64 warps
// per quarter, lane = p mod 32), so every read of the token vectors (k, q,
// alpha) is a single-address broadcast, and the state rows it moves are
// contiguous.  The reductions over rows (S'^T k, S'^T q) are summed over the
// quarters through shared memory: one block barrier per token, the partial
// sums double-buffered by token parity.  The token vectors (k, q, alpha, v,
// q . k, beta) are prepared once per batch of 8 tokens into shared memory,
// one warp per token.
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kTokBatch = 8;

// 16-byte shared-memory load, issued where it stands: the compiler neither
// merges it with an earlier load of the same address nor hoists it (holding
// a whole token's vectors in registers next to the state would spill)
__device__ __forceinline__ float4 lds128_fresh(const float* p) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// bulk asynchronous copy global -> shared (16-byte aligned, size a multiple of
// 16), completion counted in bytes on the mbarrier
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%2], [%3], %1, [%0];"
      ::"r"(smem_addr(bar)), "r"(bytes), "r"(smem_addr(dst)), "l"(src)
      : "memory");
}

// The state of unit u into shared memory; in the bounds-checked build a copy
// whose source range is outside the state buffer is not issued, and a plain
// arrival completes the phase instead (the unit then computes from stale data,
// and the device error word reports the violation)
template <int D>
__device__ __forceinline__ void fetch_state(float* dst, float* S, int64_t u, int64_t units,
                                            uint64_t* bar, int* err) {
  if (kda_guard(u * D * D, static_cast<int64_t>(D) * D, units * D * D, err))
    bulk_load(dst, S + u * D * D, static_cast<uint32_t>(D * D * 4), bar);
  else
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded wait on the mbarrier phase `parity`: false after `limit` polls (each
// poll blocks for a hardware-chosen interval), never an endless spin.
__device__ __forceinline__ bool wait_parity(uint64_t* bar, uint32_t parity,
                                            uint32_t limit = 1u << 22) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// PER (4 or 2) consecutive bf16 / f32 values with one vector load
template <int PER>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float (&f)[PER]) {
  if constexpr (PER == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(u << 16); f[1] = __uint_as_float(u & 0xffff0000u);
  }
}
template <int PER>
__device__ __forceinline__ void load_f32(const float* p, float (&f)[PER]) {
  if constexpr (PER == 4) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
  } else {
    const float2 u = *reinterpret_cast<const float2*>(p);
    f[0] = u.x; f[1] = u.y;
  }
}

template <int D>
struct TokCfg {
  static constexpr int kThreads = 2 * D;
  static constexpr int kCtasPerSm = D == 128 ? 2 : 4;  // 64 KiB | 16 KiB of state each
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kRows = D / 4;   // state rows per thread (2 columns each)
  static constexpr int kWarpsPerQuarter = D / 64;
  // dynamic shared memory: state buffer, token vectors (k P, q P, k / P, v, P),
  // partial sums [parity][a | b][quarter][D], scalars, mbarrier
  static constexpr size_t kStateBytes = static_cast<size_t>(D) * D * 4;
  static constexpr size_t kVecBytes = 5 * kTokBatch * D * 4;
  static constexpr size_t kPartBytes = 2 * 2 * 4 * D * 4;
  static constexpr size_t kSmem = kStateBytes + kVecBytes + kPartBytes + 2 * kTokBatch * 4 + 16;
};

template <int D, bool FUSED>
__global__ void __launch_bounds__(TokCfg<D>::kThreads, TokCfg<D>::kCtasPerSm)
decode_tokens_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                     const uint16_t* __restrict__ v, const float* __restrict__ log_alpha,
                     const uint16_t* __restrict__ gate, const float* __restrict__ beta,
                     float* __restrict__ S, uint16_t* __restrict__ out,
                     const int32_t* __restrict__ commit, int32_t K, int32_t H, int64_t units,
                     int* __restrict__ err) {
  using Cfg = TokCfg<D>;
  constexpr int RPT = Cfg::kRows, WPQ = Cfg::kWarpsPerQuarter;
  extern __shared__ __align__(128) unsigned char dsm[];
  float* s_state = reinterpret_cast<float*>(dsm);                          // [D][D]
  float(*s_kp)[D] = reinterpret_cast<float(*)[D]>(dsm + Cfg::kStateBytes);  // [batch][D]: k P
  float(*s_qp)[D] = s_kp + kTokBatch;  // q P
  float(*s_ki)[D] = s_qp + kTokBatch;  // k / P (alpha until the running product is formed)
  float(*s_v)[D] = s_ki + kTokBatch;
  float(*s_P)[D] = s_v + kTokBatch;    // P after token tt of the batch
  float(*s_part)[4][D] =  // [parity * 2 + (0: S'^T k | 1: S'^T q)][quarter][column]
      reinterpret_cast<float(*)[4][D]>(dsm + Cfg::kStateBytes + Cfg::kVecBytes);
  float* s_qk = reinterpret_cast<float*>(dsm + Cfg::kStateBytes + Cfg::kVecBytes + Cfg::kPartBytes);
  float* s_beta = s_qk + kTokBatch;
  uint64_t* bar = reinterpret_cast<uint64_t*>(s_beta + kTokBatch);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp / WPQ, j = 2 * (32 * (warp % WPQ) + lane);  // columns j, j + 1
  const int64_t stride = gridDim.x;

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  int64_t unit = blockIdx.x;  // sequence * H + head
  if (tid == 0 && unit < units) fetch_state<D>(s_state, S, unit, units, bar, err);
  uint32_t parity = 0;

#pragma unroll 1
  for (; unit < units; unit += stride) {
    const int64_t n = unit / H, h = unit % H;
    // ---- this unit's state: wait for its copy, take it into registers
    const bool arrived = wait_parity(bar, parity);
    parity ^= 1u;
    float2 st[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      st[i] = arrived ? *reinterpret_cast<const float2*>(s_state + (quarter * RPT + i) * D + j)
                      : make_float2(0.f, 0.f);
    // every thread has its state, so the buffer can take the next unit's; and
    // every thread agrees whether the copy arrived
    if (__syncthreads_or(!arrived)) {  // it never completed: report, and stop this CTA
      if (tid == 0) atomicOr(err, kDevErrTimeout);
      return;
    }
    if (tid == 0 && unit + stride < units) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fetch_state<D>(s_state, S, unit + stride, units, bar, err);
    }

    int n_commit = K;
    if (commit) {
      if (!kda_guard(n, 1, units / H, err)) continue;
      n_commit = commit[n];
      if (n_commit < 0 || n_commit > K) {  // rejected: nothing is written for this unit
        if (tid == 0) atomicOr(err, kDevErrCommit);
        continue;
      }
    }
    float* Sc = S + unit * D * D + static_cast<int64_t>(quarter * RPT) * D + j;

#pragma unroll 1
    for (int t0 = 0; t0 < K; t0 += kTokBatch) {
      const int kb = min(kTokBatch, K - t0);
      // ---- token vectors of the batch: warp w prepares tokens w, w + kWarps, ...
#pragma unroll 1
      for (int tt = warp; tt < kb; tt += Cfg::kWarps) {
        const int64_t row = (n * K + t0 + tt) * H + h;
        constexpr int PER = D / 32;  // channels per lane: lane * PER .. + PER - 1 (4 or 2)
        float kf[PER], qf[PER], al[PER], vf[PER];
        const int64_t e0 = row * D + lane * PER;  // one vector load per input
        if (!kda_guard(e0, PER, units * K * D, err)) continue;  // warp-uniform
        load_bf16<PER>(k + e0, kf);
        load_bf16<PER>(q + e0, qf);
        load_bf16<PER>(v + e0, vf);
        if (FUSED) {
          load_bf16<PER>(gate + e0, al);
#pragma unroll
          for (int x = 0; x < PER; ++x) al[x] = expf(gate_log_alpha(al[x]));
        } else {
          load_f32<PER>(log_alpha + e0, al);
#pragma unroll
          for (int x = 0; x < PER; ++x) al[x] = expf(clamp_log_alpha(al[x]));
        }
        if (FUSED) {  // L2-normalise q and k, then round them to bf16
          float sk = 0.f, sq = 0.f;
#pragma unroll
          for (int x = 0; x < PER; ++x) { sk += kf[x] * kf[x]; sq += qf[x] * qf[x]; }
#pragma unroll
          for (int o = 16; o; o >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
          }
          const float ck = l2_scale(sk), cq = l2_scale(sq);
#pragma unroll
          for (int x = 0; x < PER; ++x) {
            kf[x] = bf16_to_f32(f32_to_bf16(kf[x] * ck));
            qf[x] = bf16_to_f32(f32_to_bf16(qf[x] * cq));
          }
        }
        float qk = 0.f;
#pragma unroll
        for (int x = 0; x < PER; ++x) {
          const int c = lane * PER + x;
          s_kp[tt][c] = kf[x];
          s_qp[tt][c] = qf[x];
          s_ki[tt][c] = al[x];
          s_v[tt][c] = vf[x];
          qk += qf[x] * kf[x];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);
        if (lane == 0) {
          s_qk[tt] = qk;
          s_beta[tt] = kda_guard(row, 1, units * K, err) ? beta[row] : 0.f;
        }
      }
      __syncthreads();
      if (tid < D) {  // running products of alpha over the batch, per key channel
        float P = 1.f;
        for (int tt = 0; tt < kb; ++tt) {
          P *= s_ki[tt][tid];
          const float kc = s_kp[tt][tid];
          s_P[tt][tid] = P;
          s_kp[tt][tid] = kc * P;
          s_qp[tt][tid] *= P;
          s_ki[tt][tid] = kc / P;
        }
      }
      __syncthreads();

      // ---- the batch's tokens, in order
#pragma unroll 1
      for (int tt = 0; tt < kb; ++tt) {
        const int t = t0 + tt;
        const int64_t row = (n * K + t) * H + h;
        const float2 vt = *reinterpret_cast<const float2*>(&s_v[tt][j]);
        const float* kk = &s_kp[tt][quarter * RPT];
        const float* qq = &s_qp[tt][quarter * RPT];
        const float* ki = &s_ki[tt][quarter * RPT];
        // a = (S'^T k)_{j, j+1}, b = (S'^T q)_{j, j+1}: packed two-lane
        // multiply-adds (each lane rounds exactly as a scalar fmaf would)
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; i += 4) {
          const float4 k4 = lds128_fresh(kk + i);
          const float4 q4 = lds128_fresh(qq + i);
          const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            a = __ffma2_rn(make_float2(kv[x], kv[x]), st[i + x], a);
            b = __ffma2_rn(make_float2(qv[x], qv[x]), st[i + x], b);
          }
        }
        // sum over the four quarters, in quarter order (every thread of a
        // column pair gets the same sums)
        const int par = 2 * (t & 1);
        *reinterpret_cast<float2*>(&s_part[par][quarter][j]) = a;
        *reinterpret_cast<float2*>(&s_part[par + 1][quarter][j]) = b;
        __syncthreads();
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 pa = *reinterpret_cast<const float2*>(&s_part[par][x][j]);
          const float2 pb = *reinterpret_cast<const float2*>(&s_part[par + 1][x][j]);
          a0 += pa.x; a1 += pa.y; b0 += pb.x; b1 += pb.y;
        }
        const float u0 = s_beta[tt] * (vt.x - a0), u1 = s_beta[tt] * (vt.y - a1);
        if (quarter == 0 && kda_guard(row * D + j, 2, units * K * D, err))
          *reinterpret_cast<uint32_t*>(out + row * D + j) =
              static_cast<uint32_t>(f32_to_bf16(b0 + s_qk[tt] * u0)) |
              (static_cast<uint32_t>(f32_to_bf16(b1 + s_qk[tt] * u1)) << 16);
        const float2 u = make_float2(u0, u1);
#pragma unroll
        for (int i = 0; i < RPT; i += 4) {
          const float4 k4 = lds128_fresh(ki + i);
          const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) st[i + x] = __ffma2_rn(make_float2(kv[x], kv[x]), u, st[i + x]);
        }
        if (t + 1 == n_commit) {  // S = P Z
          const float* pp = &s_P[tt][quarter * RPT];
#pragma unroll
          for (int i = 0; i < RPT; i += 4) {
            const float4 p4 = lds128_fresh(pp + i);
            const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int x = 0; x < 4; ++x)
              if (kda_guard(unit * D * D + static_cast<int64_t>(quarter * RPT + i + x) * D + j, 2,
                            units * D * D, err))
                __stcs(reinterpret_cast<float2*>(Sc + static_cast<int64_t>(i + x) * D),
                       __fmul2_rn(st[i + x], make_float2(pv[x], pv[x])));
          }
        }
      }
      if (t0 + kTokBatch < K) {  // back to S for the next batch
        const float* pp = &s_P[kb - 1][quarter * RPT];
#pragma unroll
        for (int i = 0; i < RPT; i += 4) {
          const float4 p4 = lds128_fresh(pp + i);
          const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) st[i + x] = __fmul2_rn(st[i + x], make_float2(pv[x], pv[x]));
        }
      }
      __syncthreads();  // the next batch (or unit) rewrites the token vectors
    }
  }
  // A CTA leaves only after the wait for its last issued copy (the loop's
  // last iteration issues none), so no copy into its shared memory is pending.
}

template <int D, bool FUSED>
cudaError_t launch_t(const DecodeArgs& a, int64_t units, cudaStream_t s) {
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  auto kern = decode_tokens_kernel<D, FUSED>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(TokCfg<D>::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t per_wave = static_cast<int64_t>(TokCfg<D>::kCtasPerSm) * sms[dev];
  const int64_t grid = units < per_wave ? units : per_wave;
  kern<<<static_cast<unsigned>(grid), TokCfg<D>::kThreads, TokCfg<D>::kSmem, s>>>(
      a.q, a.k, a.v, a.log_alpha, a.gate, a.beta, a.S, a.out, a.commit, a.K, a.H, units, a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tokens(const DecodeArgs& a, cudaStream_t s) {
  const int64_t units = static_cast<int64_t>(a.N) * a.H;
  if (units == 0) return cudaSuccess;
  prof_begin(s, "kda_decode_tokens");
  const bool fused = a.gate != nullptr;
  cudaError_t e;
  if (a.dk == 128)
    e = fused ? launch_t<128, true>(a, units, s) : launch_t<128, false>(a, units, s);
  else
    e = fused ? launch_t<64, true>(a, units, s) : launch_t<64, false>(a, units, s);
  prof_end(s, "kda_decode_tokens");
  return e;
}

}  // namespace kda
