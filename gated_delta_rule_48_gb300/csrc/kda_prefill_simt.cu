// Chunk-parallel prefill on the CUDA cores (fp32 throughout).
//
// One CTA owns one unit = (segment, head, block of 64 state columns) and walks
// the segment's 64-token chunks in order, keeping its dk x 64 block of the
// state in shared memory.  Per chunk (tokens r, i inside the chunk,
// g = within-chunk cumulative clamped log-decay per key channel):
//
//   A_kk[r,i] = beta_r sum_c k_rc k_ic e^{g_rc - g_ic}   (i <  r)
//   A_qk[r,i] =        sum_c q_rc k_ic e^{g_rc - g_ic}   (i <= r)
//   U  = (I + A_kk)^{-1} Diag(beta) (V - (k * e^g) S)      forward substitution
//   O  = (q * e^g) S + A_qk U                              -> out
//   S <- Diag(e^{g_last}) S + (k * e^{g_last - g})^T U
//
// This is the chunked form of the recurrence: tokens of a chunk are handled
// together and only the state passes between chunks (meridianbulletin.com
// article, section "Parallelizing Sequential State Updates").  Differences
// of cumulative log-decays are taken before exponentiating, so every exponent
// above is <= 0 and nothing can overflow.
//
// Columns of the state are independent given the chunk's k, q, gates, so the
// 64-column blocks run in separate CTAs.  In the summary pass of a split
// sequence the unit's columns are either value columns started from zero
// (they accumulate the segment's increment B) or identity columns with zero
// values (they accumulate its transition M); see kda_plan.cu.
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

namespace {

constexpr int C = kChunk;      // 64
constexpr int NB = 64;         // state columns per CTA
constexpr int kThreads = 256;

template <int D>
struct SimtSmem {
  static constexpr int LD = D + 1;  // padded row stride of token x channel arrays
  float k[C * LD];
  float q[C * LD];
  float g[C * LD];
  float w[C * LD];    // k e^g, then q e^g, then k e^{g_last - g}
  float v[C * NB];    // values, then U
  float akk[C * C];
  float aqk[C * C];
  float S[D * NB];
  float x[C * NB];    // right-hand side of the triangular solve
  float beta[C];
  float glast[D];
};

// mode 0 = summary (B | M columns of non-final segments), 1 = replay.
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(PrefillArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<D>& sm = *reinterpret_cast<SimtSmem<D>*>(smem_raw);
  constexpr int LD = SimtSmem<D>::LD;
  const int tid = threadIdx.x;
  const int32_t seg_id = blockIdx.x;
  const int h = blockIdx.y;
  const int cb = blockIdx.z;
  if (seg_id >= *a.plan.n_segs) return;
  const Segment sg = a.plan.segs[seg_id];
  const bool last = sg.index + 1 == sg.count;
  if (MODE == 0 && last) return;  // the last segment of a sequence needs no summary

  const int H = a.H, DV = a.dv;
  const int vblocks = DV / NB;
  // column kind: value columns [col0, col0 + NB) of v / S, or identity columns
  const bool ident = MODE == 0 && cb >= vblocks;
  const int col0 = ident ? (cb - vblocks) * NB : cb * NB;

  // ---- initial state block
  for (int i = tid; i < D * NB; i += kThreads) {
    const int c = i / NB, j = i % NB;
    float s0 = 0.f;
    if (MODE == 0) {
      s0 = ident ? (c == col0 + j ? 1.f : 0.f) : 0.f;
    } else if (sg.index == 0) {
      if (a.S0) s0 = a.S0[((static_cast<int64_t>(sg.seq) * H + h) * D + c) * DV + col0 + j];
    } else {
      s0 = a.entry_state[((static_cast<int64_t>(seg_id) * H + h) * D + c) * DV + col0 + j];
    }
    sm.S[i] = s0;
  }

  // State checkpoints (replay): tokens of the sequence before this segment
  const int64_t ckpt_ci = (MODE == 1 && a.ckpt) ? a.plan.ckpt_interval : 0;
  const int64_t seq_t0 = ckpt_ci > 0 ? a.plan.segs[sg.first].t0 : 0;

  for (int64_t c0 = sg.t0; c0 < sg.t1; c0 += C) {
    const int valid = sg.t1 - c0 < C ? static_cast<int>(sg.t1 - c0) : C;
    __syncthreads();
    // ---- load the chunk; rows past the segment end act as identity tokens
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      float kk = 0.f, qq = 0.f, la = 0.f;
      if (r < valid) {
        const int64_t idx = ((c0 + r) * H + h) * D + c;
        kk = bf16_to_f32(a.k[idx]);
        if (MODE == 1) qq = bf16_to_f32(a.q[idx]);
        la = a.fused ? gate_log_alpha(bf16_to_f32(a.gate[idx])) : clamp_log_alpha(a.log_alpha[idx]);
      }
      sm.k[r * LD + c] = kk;
      sm.q[r * LD + c] = qq;
      sm.g[r * LD + c] = la;
    }
    for (int i = tid; i < C * NB; i += kThreads) {
      const int r = i / NB, j = i % NB;
      float vv = 0.f;
      if (r < valid && !ident) vv = bf16_to_f32(a.v[((c0 + r) * H + h) * DV + col0 + j]);
      sm.v[i] = vv;
    }
    for (int r = tid; r < C; r += kThreads)
      sm.beta[r] = r < valid ? a.beta[(c0 + r) * H + h] : 0.f;
    __syncthreads();
    if (a.fused) {  // raw q, k: L2-normalise each token's row, round to bf16
      for (int rr = tid; rr < 2 * C; rr += kThreads) {
        if (rr >= C && MODE != 1) break;
        float* row = (rr < C ? sm.k : sm.q) + (rr % C) * LD;
        float ss = 0.f;
        for (int c = 0; c < D; ++c) ss += row[c] * row[c];
        const float sc = l2_scale(ss);
        for (int c = 0; c < D; ++c) row[c] = bf16_to_f32(f32_to_bf16(row[c] * sc));
      }
      __syncthreads();
    }

    // ---- cumulative log-decay per channel
    for (int c = tid; c < D; c += kThreads) {
      float run = 0.f;
      for (int r = 0; r < C; ++r) {
        run += sm.g[r * LD + c];
        sm.g[r * LD + c] = run;
      }
      sm.glast[c] = run;
    }
    __syncthreads();

    // ---- A_kk (and A_qk in replay); k e^g into w
    for (int i = tid; i < C * C; i += kThreads) {
      const int r = i / C, ii = i % C;
      float akk = 0.f, aqk = 0.f;
      if (ii <= r) {
        for (int c = 0; c < D; ++c) {
          const float e = __expf(sm.g[r * LD + c] - sm.g[ii * LD + c]) * sm.k[ii * LD + c];
          akk += sm.k[r * LD + c] * e;
          if (MODE == 1) aqk += sm.q[r * LD + c] * e;
        }
      }
      sm.akk[i] = ii < r ? sm.beta[r] * akk : 0.f;
      if (MODE == 1) sm.aqk[i] = aqk;
    }
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      sm.w[r * LD + c] = sm.k[r * LD + c] * __expf(sm.g[r * LD + c]);
    }
    __syncthreads();

    // ---- right-hand side beta (V - (k e^g) S)
    for (int i = tid; i < C * NB; i += kThreads) {
      const int r = i / NB, j = i % NB;
      float acc = 0.f;
      for (int c = 0; c < D; ++c) acc += sm.w[r * LD + c] * sm.S[c * NB + j];
      sm.x[i] = sm.beta[r] * (sm.v[i] - acc);
    }
    __syncthreads();

    // ---- U = (I + A_kk)^{-1} x : forward substitution, 4 lanes per column
    {
      const int j = tid >> 2, p = tid & 3;  // 64 columns x 4 partial lanes
      for (int r = 0; r < C; ++r) {
        float part = 0.f;
        for (int ii = p; ii < r; ii += 4) part += sm.akk[r * C + ii] * sm.v[ii * NB + j];
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (p == 0) sm.v[r * NB + j] = sm.x[r * NB + j] - part;
        __syncwarp();
      }
    }
    __syncthreads();

    // ---- O = (q e^g) S + A_qk U  (replay only)
    if (MODE == 1) {
      for (int i = tid; i < C * D; i += kThreads) {
        const int r = i / D, c = i % D;
        sm.w[r * LD + c] = sm.q[r * LD + c] * __expf(sm.g[r * LD + c]);
      }
      __syncthreads();
      for (int i = tid; i < C * NB; i += kThreads) {
        const int r = i / NB, j = i % NB;
        if (r >= valid) continue;
        float acc = 0.f;
        for (int c = 0; c < D; ++c) acc += sm.w[r * LD + c] * sm.S[c * NB + j];
        for (int ii = 0; ii <= r; ++ii) acc += sm.aqk[r * C + ii] * sm.v[ii * NB + j];
        a.out[((c0 + r) * H + h) * DV + col0 + j] = f32_to_bf16(acc);
      }
      __syncthreads();
    }

    // ---- S <- Diag(e^{g_last}) S + (k e^{g_last - g})^T U
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      sm.w[r * LD + c] = sm.k[r * LD + c] * __expf(sm.glast[c] - sm.g[r * LD + c]);
    }
    __syncthreads();
    for (int i = tid; i < D * NB; i += kThreads) {
      const int c = i / NB, j = i % NB;
      float acc = __expf(sm.glast[c]) * sm.S[i];
      for (int r = 0; r < C; ++r) acc += sm.w[r * LD + c] * sm.v[r * NB + j];
      sm.S[i] = acc;
      if (ckpt_ci > 0) {  // the state after this chunk, if the sequence has a checkpoint here
        const int64_t pos = c0 + valid - seq_t0;
        if (pos % ckpt_ci == 0) {
          const int64_t slot = a.plan.ckpt_base[sg.seq] + pos / ckpt_ci - 1;
          if (slot < a.plan.ckpt_max)
            a.ckpt[((slot * H + h) * D + c) * static_cast<int64_t>(DV) + col0 + j] = acc;
        }
      }
    }
  }
  __syncthreads();

  // ---- write back
  if (MODE == 0) {
    const int W = DV + D;
    const int colw = ident ? DV + col0 : col0;
    float* rec = a.incr_trans + (static_cast<int64_t>(seg_id) * H + h) * static_cast<int64_t>(D) * W;
    for (int i = tid; i < D * NB; i += kThreads) {
      const int c = i / NB, j = i % NB;
      rec[static_cast<int64_t>(c) * W + colw + j] = sm.S[i];
    }
  } else if (last && a.S_final) {
    float* sf = a.S_final + (static_cast<int64_t>(sg.seq) * H + h) * static_cast<int64_t>(D) * DV;
    for (int i = tid; i < D * NB; i += kThreads) {
      const int c = i / NB, j = i % NB;
      sf[static_cast<int64_t>(c) * DV + col0 + j] = sm.S[i];
    }
  }
}

template <int D, int MODE>
cudaError_t launch_simt(const PrefillArgs& a, cudaStream_t s, const char* name) {
  const size_t smem = sizeof(SimtSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(prefill_simt_kernel<D, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int blocks = MODE == 0 ? (a.dv + D) / NB : a.dv / NB;
  dim3 grid(a.plan.capacity, a.H, blocks);
  prof_begin(s, name);
  prefill_simt_kernel<D, MODE><<<grid, kThreads, smem, s>>>(a);
  prof_end(s, name);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_summary(const PrefillArgs& a, cudaStream_t s) {
  return a.dk == 128 ? launch_prefill_summary_tc(a, s)
                     : launch_simt<64, 0>(a, s, "kda_prefill_summary");
}

cudaError_t launch_prefill_replay(const PrefillArgs& a, cudaStream_t s) {
  return a.dk == 128 ? launch_prefill_replay_tc(a, s)
                     : launch_simt<64, 1>(a, s, "kda_prefill_replay");
}

}  // namespace kda
