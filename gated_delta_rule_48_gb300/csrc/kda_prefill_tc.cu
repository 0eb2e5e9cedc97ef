// Chunk-parallel prefill on the tcgen05 tensor cores (dk = dv = 128; 64 runs
// zero-padded to 128).
//
// One CTA per unit = (segment, head) walks the segment's 64-token chunks in
// order.  The state is kept TRANSPOSED in tensor memory
// (S^T: lane = value channel j, column = key channel c, fp32) for the whole
// segment and is itself the A operand of the MMAs that read it, so it never
// leaves the SM between chunks.  Per chunk (tokens r, i of the chunk, g the
// within-chunk cumulative clamped log-decay per key channel):
//
//   strip products (bf16):  A_qk[r,i] = sum_c q_rc k_ic e^{g_rc - g_ic}  (i <= r)
//                           A_kk[r,i] = beta_r sum_c k_rc k_ic e^{g_rc - g_ic}  (i < r)
//   UT transform (fp32):    T = (I + A_kk)^{-1} Diag(beta)
//   U~^T = V^T T^T (bf16 hi + lo)
//   hand-off (tf32):        replay:  P^T = S^T (k e^g)^T,  U^T = U~^T - P^T T^T
//                           summary: W^T = (k e^g)^T T^T,  U^T = U~^T - S^T W^T
//                           O^T = S^T (q e^g)^T + U^T A_qk^T        -> out (replay)
//                           S^T <- S^T Diag(e^{g_last}) + U^T K',  K' = k e^{g_last - g}
//
// Tokens of a chunk are processed together and only the state is handed on
// (meridianbulletin.com article, section "Parallelizing Sequential State
// Updates").  The decay inside a chunk enters the strip products through a
// per-strip anchor G: q_r e^{g_r - G} against k_i e^{G - g_i}.  The chunk has
// two 32-token strips anchored at their middle token, so every token is at
// most 16 steps from its anchor and, with log-decay >= -5 per step, every
// factor lies in [e^-80, e^80] -- finite in bf16 and fp32.  This is the
// bound of the orkas.ai close read (section "A lower bound that deleted a
// GPU code path": accumulated log-decay over 16 tokens stays within (-80, 0),
// so the reciprocal stays under e^80 and the diagonal tiles can use the same
// dense matrix multiply as the rest), applied on both sides of the anchor.
//
// Operand precision: strip products in bf16 (their error only perturbs T and
// the output); T is fp32 and enters the tf32 MMA rounded to nearest, and the
// bf16 MMA with V (exact in bf16) as a hi + lo pair of bf16; every operand on
// the state path is tf32 rounded to nearest; the two output-only operands
// (q e^g and A_qk) are stored fp32 and read by the tensor core as tf32, i.e.
// truncated; accumulation is fp32.  tf32
// operands are always laid out K-major: K' (and, for W^T, k e^g) are written
// transposed, [key channel][token]; k e^g for P^T and q e^g [token][channel].
//
// Schedule of chunk n in the replay (16 worker warps; two issuer threads in a
// control warpgroup issue the MMAs and the TMA copies):
//   A  strip MMA (n) ; P^T (n)           || read O^T (n-1) out of TMEM -> out
//   B  strip read-out, UT transform (in place), T to SMEM; meanwhile -P^T
//      rounded to tf32 in TMEM and q e^g to SMEM
//   C  O^T = S^T (q e^g)^T ; U^T = U~^T - P^T T^T  || K' (n), decay scan of n+1
//   F  decay the columns of S^T, round U^T to tf32 (in TMEM)
//   G  O^T += U^T A_qk^T ; S^T += U^T K' || operands of chunk n+1 to SMEM
// The summary runs C as W^T, U~^T || K', then D (-W to SMEM) and E (U^T -=
// S^T W^T for both of its states || decay scan of n+1).
// Raw q, k, log_alpha stream in by TMA one chunk ahead; v after step C.
//
// Split prefill: every chunk's T is the same whether the summary or the
// replay of its segment computes it (the key rows of the strip products do
// not depend on the query rows).  So the summary keeps each T (tf32 copy and
// bf16 hi / lo, 32 KiB) in the workspace with one bulk store, and the second
// pass's replay of a summarised segment (TIN) runs B as: T loaded by one bulk
// copy into the strip operand's buffer once the strip MMA has read it, only
// the query rows read out, -P^T rounded on all 16 warps.  Its outputs are
// bit for bit those of a replay that computes T.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

namespace {

using namespace sm100;

constexpr int D = 128;          // dk = dv
constexpr int C = kChunk;       // 64
constexpr int kWorkers = 512;                 // 16 worker warps
constexpr int kWarps = kWorkers / 32;
constexpr int kThreads = kWorkers + 128;      // + 1 control warpgroup (2 MMA issuers)
constexpr uint32_t kTmemCols = 512;
// Registers: launched at kLaunchRegs per thread (5 warps share a sub-partition);
// the control warpgroup then hands part of its share to the workers (setmaxnreg).
constexpr uint32_t kLaunchRegs = 96, kWorkerRegs = 104, kCtrlRegs = 64;
static_assert(kWorkers * kWorkerRegs + 128 * kCtrlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");

// TMEM column map (fp32 columns; 128 lanes)
constexpr uint32_t kColS = 0;     // S^T            128 columns
constexpr uint32_t kColA = 128;   // strip products  96 columns
constexpr uint32_t kColW = 256;   // W^T             64 columns (lane = key channel)
constexpr uint32_t kColU = 320;   // U^T             64 columns (lane = value channel)
constexpr uint32_t kColO = 384;   // O^T             64 columns

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kRawQ = 0;                 // bf16 [64][128] sw128 (2 blocks)
constexpr uint32_t kRawK = kRawQ + 16384;
constexpr uint32_t kRawV = kRawK + 16384;
constexpr uint32_t kRawL = kRawV + 16384;     // f32 [64][128] sw128 (4 blocks)
constexpr uint32_t kR = kRawL + 32768;        // phase-dependent operand region (72 KiB):
//   operands: strip A bf16 [128][128] at +0, strip B bf16 [96][128] at +32768
//   UT:       T tf32 [64][64] at +0, T_hi / T_lo bf16 [64][64] at +16384 / +24576,
//             A_kk -> T' f32 [64][kLdA] at +32768, scratch 32 x 36 f32 after it
//             (the transposed block A_(10) sits in the then idle K' buffer)
//   always:   A_qk tf32 [64][64] at +57344 (replay)
constexpr uint32_t kLdA = 68;                 // padded row stride (floats)
constexpr uint32_t kRT = 0, kRTh = 16384, kRTl = 24576, kRAkk = 32768;
constexpr uint32_t kRAqk = 57344;
constexpr uint32_t kRXs = kRAkk + C * kLdA * 4;  // UT scratch, 32 x 36 f32
constexpr uint32_t kKG = kR + 73728;          // k e^g tf32: replay [token][channel] -> q e^g;
                                              // summary transposed -> -W
constexpr uint32_t kKP = kKG + 32768;         // K' (transposed)            tf32
constexpr uint32_t kMisc = kKP + 32768;
// f32 warp totals [16][128] of the decay scan, then their exclusive prefixes:
// live only inside the scan, in a part of R that no operand uses then
constexpr uint32_t kTot = kR + 40960;
constexpr uint32_t kG0 = kMisc;              // strip anchors g_15, g_47 [128] each
constexpr uint32_t kG1 = kG0 + 512;
constexpr uint32_t kEGl = kG1 + 512;          // e^{g_last} [2][128], by chunk parity
constexpr uint32_t kPC = kEGl + 1024;         // per-channel factors [5][128]: e^{G0}, e^{G1},
                                              // e^{g_last - G0}, e^{g_last - G1}, e^{G1 - G0}
constexpr uint32_t kBeta = kPC + 5 * 512;
constexpr uint32_t kBars = kBeta + 256;       // 13 mbarriers, TMEM slot, abort flag
constexpr uint32_t kSmemBytes = kBars + 128 + 1024;  // + alignment slack
static_assert(kRXs + 32 * 36 * 4 <= kRAqk, "UT scratch overlaps A_qk");
static_assert(kTot >= kR + 32768 && kTot + kWarps * 512 <= kR + kRAqk, "scan totals placement");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(13 * 8 + 2 * 4 <= 128, "mbarriers, TMEM slot and abort flag");

struct TcMaps {
  CUtensorMap q, k, v, la;  // la: f32 log alpha, or the bf16 gate logits when fused
};

enum : int { kModeSummary = 0, kModeReplay = 1 };

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Barrier among the 16 worker warps only (the control warps never join it).
__device__ __forceinline__ void worker_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Packed two-lane fp32 arithmetic (each lane rounds exactly as the scalar
// operation would): half the instructions of the scalar form.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 bcast2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  return __fadd2_rn(a, make_float2(-b.x, -b.y));
}
// 4 bf16 (two 32-bit words) -> channels 0, 1 and 2, 3 as float2 pairs
__device__ __forceinline__ void unpack4x2(uint2 u, float2& f01, float2& f23) {
  f01 = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
  f23 = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ uint2 pack4x2_bf16(float2 f01, float2 f23) {
  return make_uint2(pack_bf16x2(f01.x, f01.y), pack_bf16x2(f23.x, f23.y));
}
__device__ __forceinline__ uint4 pack4x2_tf32(float2 f01, float2 f23) {
  return make_uint4(f32_to_tf32_rn(f01.x), f32_to_tf32_rn(f01.y), f32_to_tf32_rn(f23.x),
                    f32_to_tf32_rn(f23.y));
}
__device__ __forceinline__ float2 rcp2(float2 a) { return make_float2(rcp_approx(a.x), rcp_approx(a.y)); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

__device__ __forceinline__ void unpack4(uint2 u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}
// Fused input preparation.  The 8 vectors k_r, q_r of a warp's 4 tokens each
// span the warp (4 channels per lane); each is scaled to unit L2 norm,
// x / max(||x||, 1e-12), and rounded to bf16.  The 8 sums of squares are
// reduced together: three exchange steps halve the set each time (4 + 2 + 1
// shuffles), two more finish one sum per lane (vector 4 * bit4 + 2 * bit3 +
// bit2 of the lane), and 8 shuffles from lanes 4j hand the scales back --
// 17 shuffles instead of 40.  Every lane of the warp must call it.
__device__ __forceinline__ void l2norm8_bf16(uint2 (&kr)[4], uint2 (&qr)[4], int lane) {
  float f[8][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint2 a = kr[i], b = qr[i];
    f[i][0] = __uint_as_float(a.x << 16); f[i][1] = __uint_as_float(a.x & 0xffff0000u);
    f[i][2] = __uint_as_float(a.y << 16); f[i][3] = __uint_as_float(a.y & 0xffff0000u);
    f[4 + i][0] = __uint_as_float(b.x << 16); f[4 + i][1] = __uint_as_float(b.x & 0xffff0000u);
    f[4 + i][2] = __uint_as_float(b.y << 16); f[4 + i][3] = __uint_as_float(b.y & 0xffff0000u);
  }
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    v[j] = f[j][0] * f[j][0] + f[j][1] * f[j][1] + f[j][2] * f[j][2] + f[j][3] * f[j][3];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float w[4], x[2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float give = b4 ? v[j] : v[j + 4];
    w[j] = (b4 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, give, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float give = b3 ? w[j] : w[j + 2];
    x[j] = (b3 ? w[j + 2] : w[j]) + __shfl_xor_sync(0xffffffffu, give, 8);
  }
  float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
  y += __shfl_xor_sync(0xffffffffu, y, 2);
  y += __shfl_xor_sync(0xffffffffu, y, 1);
  const float sc_own = fminf(rsqrtf(y), 1e12f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float sc = __shfl_sync(0xffffffffu, sc_own, 4 * j);
    const uint2 o = make_uint2(pack_bf16x2(f[j][0] * sc, f[j][1] * sc),
                               pack_bf16x2(f[j][2] * sc, f[j][3] * sc));
    if (j < 4) kr[j] = o; else qr[j - 4] = o;
  }
}

// Fused input preparation: log alpha = -5 sigmoid(x) from a gate logit (the
// approximate exponential and reciprocal; e^-x = inf gives 0).
__device__ __forceinline__ float gate_log_alpha_fast(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + __expf(-x)));
  return clamp_log_alpha(-5.0f * r);
}

__device__ __forceinline__ uint4 pack4_tf32(const float (&f)[4]) {
  return make_uint4(f32_to_tf32_rn(f[0]), f32_to_tf32_rn(f[1]), f32_to_tf32_rn(f[2]),
                    f32_to_tf32_rn(f[3]));
}

// T[r][4j .. 4j+3] = f (already T'[r][c] beta_c) into the three operand copies
// of T: tf32 (rounded to nearest) [64][64] and the bf16 pair hi + lo, all
// 128-byte swizzled.  One 16-byte and two 8-byte stores.
__device__ __forceinline__ void put_T4(unsigned char* __restrict__ R, int r, int j, float4 f) {
  *reinterpret_cast<uint4*>(R + kRT + sw128_offset(C, r, 16 * j)) =
      make_uint4(f32_to_tf32_rn(f.x), f32_to_tf32_rn(f.y), f32_to_tf32_rn(f.z), f32_to_tf32_rn(f.w));
  const uint32_t h0 = pack_bf16x2(f.x, f.y), h1 = pack_bf16x2(f.z, f.w);
  const uint32_t l0 = pack_bf16x2(f.x - __uint_as_float(h0 << 16), f.y - __uint_as_float(h0 & 0xffff0000u));
  const uint32_t l1 = pack_bf16x2(f.z - __uint_as_float(h1 << 16), f.w - __uint_as_float(h1 & 0xffff0000u));
  *reinterpret_cast<uint2*>(R + kRTh + sw128_offset(C, r, 8 * j)) = make_uint2(h0, h1);
  *reinterpret_cast<uint2*>(R + kRTl + sw128_offset(C, r, 8 * j)) = make_uint2(l0, l1);
}

__device__ __forceinline__ float f4c(const float4& v, int u) {  // component u (unrolled: constant)
  return u == 0 ? v.x : u == 1 ? v.y : u == 2 ? v.z : v.w;
}

// UT transform.  sA holds a strictly lower-triangular 64 x 64 matrix A (f32,
// row stride kLdA, zero on and above the diagonal).  Computes
// T' = (I + A)^{-1} (unit lower-triangular) by doubling and writes
// T = T' Diag(beta) into its operand copies (put_T4).  Blocks of 16: D_b is
// the inverse of diagonal block b, subscripts (10), (00), (11) are 32 x 32
// halves.
//   warps 0, 1 (h = warp), with warp-level syncs only:
//     1. D_2h and D_2h+1 by forward substitution (lane = block, column),
//        in place; A is read 4 entries of a row per load;
//     2. T'_ab = -D_a (A_ab D_b) for (a, b) = (2h + 1, 2h), in place: lane =
//        (row, 8 columns), the product A_ab D_b through the scratch Xs;
//   warps 2..15 meanwhile zero T'_(01) in the copies.
//   one barrier, then
//   warps 0..7, column group q of 4 columns each (lane = row r):
//     3. X = A_(10) T'_(00) on the group's columns (A_(10) through its
//        transposed copy A10T[i][r] = A[32 + r][i]), then
//        T'_(10) = -T'_(11) X on the same columns, to T;
//   warps 8..15 meanwhile copy T'_(00) and T'_(11) to T.
// Split at its one barrier: ut_front (steps 1, 2 and the zeros), then the
// caller's worker barrier, then ut_back (step 3 and the copies).  Warps 2..15
// are free between ut_front and the barrier.
__device__ void ut_front(float* __restrict__ sA, float* __restrict__ Xs,
                         unsigned char* __restrict__ R, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 2) {
    const int h = warp;
    {
      const int b = 2 * h + (lane >> 4), j = lane & 15;
      float* Ab = sA + (16 * b) * kLdA + 16 * b;
      // row by row: x[r] = delta_rj - sum_{i < r} A[r][i] x[i], the terms in
      // the order of i (the same sums as eliminating column by column)
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int i4 = 0; i4 < r; i4 += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(Ab + r * kLdA + i4);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (i4 + u < r) acc = fmaf(-f4c(a4, u), x[i4 + u], acc);
        }
        x[r] = acc;
      }
      __syncwarp();  // both blocks of this warp are read
#pragma unroll
      for (int r = 0; r < 16; ++r) Ab[r * kLdA + j] = x[r];
    }
    __syncwarp();
    {
      const int a = 2 * h + 1, b = 2 * h;
      const int r = lane >> 1, c0 = 8 * (lane & 1);
      float* X = Xs + h * 256;  // [16][16]
      float2 acc[4];  // columns c0 + (0, 1), (2, 3), (4, 5), (6, 7)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
      const float* Arow = sA + (16 * a + r) * kLdA + 16 * b;
      const float* Db = sA + (16 * b) * kLdA + 16 * b + c0;
#pragma unroll
      for (int i4 = 0; i4 < 16; i4 += 4) {
        const float4 av = *reinterpret_cast<const float4*>(Arow + i4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 d0 = *reinterpret_cast<const float4*>(Db + (i4 + u) * kLdA);
          const float4 d1 = *reinterpret_cast<const float4*>(Db + (i4 + u) * kLdA + 4);
          const float2 s = bcast2(f4c(av, u));
          acc[0] = fma2(s, lo2(d0), acc[0]); acc[1] = fma2(s, hi2(d0), acc[1]);
          acc[2] = fma2(s, lo2(d1), acc[2]); acc[3] = fma2(s, hi2(d1), acc[3]);
        }
      }
      *reinterpret_cast<float4*>(X + r * 16 + c0) = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
      *reinterpret_cast<float4*>(X + r * 16 + c0 + 4) = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
      __syncwarp();
      const float* Da = sA + (16 * a + r) * kLdA + 16 * a;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i4 = 0; i4 < 16; i4 += 4) {
        const float4 dv = *reinterpret_cast<const float4*>(Da + i4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 x0 = *reinterpret_cast<const float4*>(X + (i4 + u) * 16 + c0);
          const float4 x1 = *reinterpret_cast<const float4*>(X + (i4 + u) * 16 + c0 + 4);
          const float2 s = bcast2(f4c(dv, u));
          acc[0] = fma2(s, lo2(x0), acc[0]); acc[1] = fma2(s, hi2(x0), acc[1]);
          acc[2] = fma2(s, lo2(x1), acc[2]); acc[3] = fma2(s, hi2(x1), acc[3]);
        }
      }
      float* Tab = sA + (16 * a + r) * kLdA + 16 * b + c0;  // A_ab was read before the last sync
      *reinterpret_cast<float4*>(Tab) = make_float4(-acc[0].x, -acc[0].y, -acc[1].x, -acc[1].y);
      *reinterpret_cast<float4*>(Tab + 4) = make_float4(-acc[2].x, -acc[2].y, -acc[3].x, -acc[3].y);
    }
  } else {
    // T'_(01) = 0: rows 0..31, columns 32..63 of the tf32 copy (256 chunks of
    // 16 bytes) and of the two bf16 copies (128 chunks each)
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int e = tid - 64; e < 512; e += 448) {
      if (e < 256) {
        *reinterpret_cast<uint4*>(R + kRT + sw128_offset(C, e >> 3, 16 * (8 + (e & 7)))) = z;
      } else {
        const int e2 = e - 256;
        *reinterpret_cast<uint4*>(R + ((e2 >> 7) ? kRTl : kRTh) +
                                  sw128_offset(C, (e2 & 127) >> 2, 64 + 16 * (e2 & 3))) = z;
      }
    }
  }
}

__device__ void ut_back(float* __restrict__ sA, float* __restrict__ Xs,
                        const float* __restrict__ A10T, const float* __restrict__ sBeta,
                        unsigned char* __restrict__ R, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 8) {
    // column group q: q = w for w < 4, 11 - w above, so each SM sub-partition
    // (warps w, w + 4) gets the same number of steps
    const int q = warp < 4 ? warp : 11 - warp;
    const int r = lane;
    float2 x01 = make_float2(0.f, 0.f), x23 = make_float2(0.f, 0.f);
    for (int i0 = 4 * q; i0 < 32; i0 += 4) {  // T'_(00)[i][4q..] = 0 for i < 4q
      float av[4];
      float4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = A10T[(i0 + u) * 32 + r];
        t[u] = *reinterpret_cast<const float4*>(sA + (i0 + u) * kLdA + 4 * q);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x01 = fma2(bcast2(av[u]), lo2(t[u]), x01);
        x23 = fma2(bcast2(av[u]), hi2(t[u]), x23);
      }
    }
    *reinterpret_cast<float4*>(Xs + r * 36 + 4 * q) = make_float4(x01.x, x01.y, x23.x, x23.y);
    __syncwarp();
    // T'_(11) is stored in full (zeros above its diagonal): 32 terms per row
    const float* T11 = sA + (32 + r) * kLdA + 32;
    float2 y01 = make_float2(0.f, 0.f), y23 = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int i0 = 0; i0 < 32; i0 += 4) {
      const float4 tv = *reinterpret_cast<const float4*>(T11 + i0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 xv = *reinterpret_cast<const float4*>(Xs + (i0 + u) * 36 + 4 * q);
        const float2 s = bcast2(f4c(tv, u));
        y01 = fma2(s, lo2(xv), y01);
        y23 = fma2(s, hi2(xv), y23);
      }
    }
    const float4 bq = *reinterpret_cast<const float4*>(sBeta + 4 * q);
    put_T4(R, 32 + r, q, make_float4(-y01.x * bq.x, -y01.y * bq.y, -y23.x * bq.z, -y23.y * bq.w));
  } else {
    // T'_(00) and T'_(11) to T: 2 halves x 32 rows x 8 column groups
    for (int e = tid - 256; e < 512; e += 256) {
      const int half = e >> 8, row = 32 * half + ((e >> 3) & 31), col = 32 * half + 4 * (e & 7);
      const float4 tv = *reinterpret_cast<const float4*>(sA + row * kLdA + col);
      const float4 bv = *reinterpret_cast<const float4*>(sBeta + col);
      put_T4(R, row, col >> 2, make_float4(tv.x * bv.x, tv.y * bv.y, tv.z * bv.z, tv.w * bv.w));
    }
  }
}

// Per-thread values of one chunk kept between steps: this thread's tokens
// 4w .. 4w+3 (w = warp) and channels 4l .. 4l+3 (l = lane).
struct ChunkRegs {
  float2 e[4][2];   // e^{g - G} (G = the strip's anchor): channels (0, 1), (2, 3)
  uint2 kraw[4];    // k (4 bf16)
  uint2 qraw[4];    // q (4 bf16)
};

// Stores 4 channel vectors (channels 4 lane + x, x = 0..3; 4 tokens each) of a
// transposed [128 channel][64 token] tf32 tile.  The order of x is rotated by
// lane so the 8 rows written by each quarter-warp differ in (row mod 8), i.e.
// land in different 16-byte swizzle slots: no bank conflicts.
__device__ __forceinline__ void st_transposed4(unsigned char* tile, int lane, int t0,
                                               const uint4 (&v)[4]) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int x = (s + (lane >> 1)) & 3;
    uint4 u = v[0];
    if (x == 1) u = v[1];
    if (x == 2) u = v[2];
    if (x == 3) u = v[3];
    *reinterpret_cast<uint4*>(tile + sw128_offset(D, 4 * lane + x, 4 * t0)) = u;
  }
}

// The same four rows without the stagger: at step s every lane writes row
// 4 lane + s.  Those stores conflict on the shared-memory banks, but the
// replay's K' measured faster this way than with the selects the stagger needs
// (the summary, whose K' and k e^g stores sit elsewhere on its chain, did not).
__device__ __forceinline__ void st_rows4(unsigned char* tile, int lane, int t0,
                                         const uint4 (&v)[4]) {
#pragma unroll
  for (int s = 0; s < 4; ++s)
    *reinterpret_cast<uint4*>(tile + sw128_offset(D, 4 * lane + s, 4 * t0)) = v[s];
}

// The (segment, head) unit of this block: one block per unit, rank-major (all
// heads of launch rank r, then rank r + 1).  The planner's order maps ranks
// to segments, longest first (the block scheduler hands out blocks in index
// order); pass 2 of a split prefill takes its own list.  False: no unit.
__device__ __forceinline__ bool unit_of(const PrefillArgs& a, int32_t& seg_id, Segment& sg,
                                        int& h) {
  const int32_t rank = static_cast<int32_t>(blockIdx.x / static_cast<uint32_t>(a.H));
  h = static_cast<int>(blockIdx.x % static_cast<uint32_t>(a.H));
  seg_id = rank;
  if (a.plan.direct_len > 0) {  // uniform batch, no planner: segment = sequence
    if (seg_id >= a.N) return false;
    sg.t0 = static_cast<int64_t>(seg_id) * a.plan.direct_len;
    sg.t1 = sg.t0 + a.plan.direct_len;
    sg.seq = seg_id;
    sg.index = 0;
    sg.count = 1;
    sg.first = seg_id;
    return true;
  }
  const int32_t* ord = a.pass == 2 ? a.plan.order2 : a.plan.order;
  const int32_t count = ord ? a.plan.n_order[a.pass == 2 ? 1 : 0] : *a.plan.n_segs;
  if (rank >= count || !kda_guard(rank, 1, a.plan.capacity, a.err)) return false;
  if (ord) seg_id = ord[rank];
  if (!kda_guard(seg_id, 1, a.plan.capacity, a.err)) return false;
  sg = a.plan.segs[seg_id];
  return true;
}

// One (segment, head) unit, in summary or replay mode (see the file header).
template <int MODE, bool FUSED, bool CKPT, bool DUMP, bool TIN = false>
__device__ __forceinline__ void prefill_tc_body(const TcMaps& maps, const PrefillArgs& a,
                                                const int32_t seg_id, const Segment& sg,
                                                const int h) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the shared array by an offset so the
  // compiler keeps every access in the shared window (32-bit addressing,
  // ld.shared / st.shared) instead of falling back to generic accesses
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool last = sg.index + 1 == sg.count;
  if (MODE == kModeSummary && last) return;
  // A summary unit carries two states through the segment: the increment B
  // (its values, from zero) and the transition M (no values, from the
  // identity).  They share the decay scan, the strip products, T, W and K';
  // only the state-reading products and the state updates are doubled.
  constexpr bool kOut = MODE == kModeReplay;
  constexpr bool kSum = MODE == kModeSummary;
  // TIN (second pass of a split prefill): a segment that the first pass
  // summarised (every one but the last of its sequence) takes each chunk's T
  // from the summary's record instead of the key-row read-out and the UT
  // transform.  The strip products still run, for A_qk.
  const bool tin = TIN && kOut && !DUMP && a.t_cache && !last;
  // Width of the caller's tensors: 128, or 64 run zero-padded to 128 (the
  // maps read channels >= 64 as zeros; zero key and query channels add
  // nothing, and zero value channels stay zero, so the 64 x 64 block is
  // exact).  Internal records (B | M, entry states) are always 128 wide.
  const int DIO = a.dv;
  // TMEM columns of this mode.  Replay: S^T 0, strip products 128, W^T 256,
  // U^T 320, O^T 384.  Summary: S_B^T 0, S_M^T 128, U_B^T 256, U_M^T 320, and
  // the strip products share 384.. with W^T: W^T of chunk n is read out (phase
  // D) before the strip MMA of chunk n+1 is issued, by the issuer that wrote it.
  constexpr uint32_t cA = kSum ? 384 : kColA;
  constexpr uint32_t cW = kSum ? 384 : kColW;
  constexpr uint32_t cU = kSum ? 256 : kColU;
  constexpr uint32_t cSM = 128, cUM = 320;  // summary only
  // Replay computes U^T = U~^T - P^T T^T with P^T = S^T (k e^g)^T (TMEM, in W^T's
  // columns): P^T needs only the state at the chunk's start and k e^g, so it
  // is issued with the strip products, and no W^T goes through SMEM.
  // Summary keeps U^T = U~^T - S^T W^T (two states' P^T would not fit TMEM).
  constexpr bool kP = kOut;
  constexpr uint32_t cP = kColW;
  const int H = a.H;
  const bool dump_unit = DUMP && seg_id == a.dump_seg && h == a.dump_head;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint64_t* bar_qkl = bars + 0;    // raw q, k, log_alpha of a chunk landed (TMA)
  uint64_t* bar_v = bars + 1;      // raw v landed (TMA)
  uint64_t* bar_done = bars + 2;   // [4] MMA group committed: 0 strip, 1 WY, 2 S-read, 3 state
  uint64_t* bar_ready = bars + 6;  // [4] operands of that group ready (one arrive per worker warp)
  uint64_t* bar_raw = bars + 10;   // raw q, k, log_alpha of a chunk read (one arrive per worker warp)
  uint64_t* bar_donep = bars + 11; // replay: P^T = S^T (k e^g)^T committed (issuer 1)
  uint64_t* bar_t = bars + 12;     // TIN replay: the chunk's T record landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 13);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  float* sTot = reinterpret_cast<float*>(sm + kTot);
  float* sG0 = reinterpret_cast<float*>(sm + kG0);
  float* sG1 = reinterpret_cast<float*>(sm + kG1);
  float* sEGl = reinterpret_cast<float*>(sm + kEGl);
  float* sBeta = reinterpret_cast<float*>(sm + kBeta);
  unsigned char* R = sm + kR;
  unsigned char* KG = sm + kKG;
  unsigned char* KP = sm + kKP;
  float* sAkk = reinterpret_cast<float*>(R + kRAkk);

  const int64_t n_chunks = (sg.t1 - sg.t0 + C - 1) / C;
  // T records of this unit: written by the summary, read by a TIN replay
  const int64_t t_base = (static_cast<int64_t>(seg_id) * H + h) * a.t_seg_chunks;
  const bool t_ok = (kSum || tin) && a.t_cache && n_chunks <= a.t_seg_chunks &&
                    kda_guard(t_base, n_chunks,
                              static_cast<int64_t>(a.plan.capacity) * H * a.t_seg_chunks, a.err);
  auto t_rec = [&](int64_t m) { return a.t_cache + (t_base + m) * kTChunkBytes; };
  // raw q (replay only), k, and log alpha (f32) or gate logits (bf16)
  const uint32_t qkl_bytes = (kOut ? 32768u : 16384u) + (FUSED ? 16384u : 32768u);
  const int quad = warp & 3, part = warp >> 2;  // TMEM lane quadrant, column quarter
  const int r0 = 4 * warp;                      // this thread's tokens r0 .. r0+3
  const int strip = warp >> 3;                  // their 32-token strip

  if (tid == 0) {
    mbar_init(bar_qkl, 1);
    mbar_init(bar_v, 1);
    for (int g = 0; g < 4; ++g) {
      mbar_init(bar_done + g, g == 0 ? 1 : 2);  // groups 1-3: one commit per issuer
      mbar_init(bar_ready + g, kWarps);
    }
    mbar_init(bar_raw, kWarps);
    mbar_init(bar_donep, 1);
    mbar_init(bar_t, 1);
    *s_abort = 0;
    if (tin && !t_ok) {  // no records for this segment (plan and workspace disagree)
      atomicOr(a.err, kDevErrCapacity);
      *s_abort = 1;
    }
    mbar_fence_init();
  }
  if (warp == kWarps) {  // the control warp owns the TMEM allocation
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  auto issue_qkl = [&](int64_t c0) {
    mbar_arrive_expect_tx(bar_qkl, qkl_bytes);
    const int32_t t = static_cast<int32_t>(c0);
    if (kOut) {
      tma_load_3d(sm + kRawQ, &maps.q, 0, h, t, bar_qkl);
      tma_load_3d(sm + kRawQ + 8192, &maps.q, 64, h, t, bar_qkl);
    }
    tma_load_3d(sm + kRawK, &maps.k, 0, h, t, bar_qkl);
    tma_load_3d(sm + kRawK + 8192, &maps.k, 64, h, t, bar_qkl);
    if (FUSED) {
      tma_load_3d(sm + kRawL, &maps.la, 0, h, t, bar_qkl);
      tma_load_3d(sm + kRawL + 8192, &maps.la, 64, h, t, bar_qkl);
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) tma_load_3d(sm + kRawL + 8192 * b, &maps.la, 32 * b, h, t, bar_qkl);
    }
  };
  auto issue_v = [&](int64_t c0) {
    mbar_arrive_expect_tx(bar_v, 16384u);
    const int32_t t = static_cast<int32_t>(c0);
    tma_load_3d(sm + kRawV, &maps.v, 0, h, t, bar_v);
    tma_load_3d(sm + kRawV + 8192, &maps.v, 64, h, t, bar_v);
  };
  auto flag_timeout = [&]() {
    atomicOr(a.err, kDevErrTimeout);
    *s_abort = 1;
  };
  // worker side: wait for MMA group g of chunk n; signal that group g's operands are ready
  // MMA group g of chunk n has completed: warp 0 alone polls its mbarrier,
  // the worker barrier then releases the other 15 warps (who would otherwise
  // each poll, taking issue slots from the warps still working)
  auto wait_done_sync = [&](int g, int64_t n) {
    if (warp == 0 && !mbar_wait(bar_done + g, static_cast<uint32_t>(n & 1))) flag_timeout();
    worker_sync();
    tc_fence_after();
  };
  auto signal_ready = [&](int g) {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_ready + g);
  };
  auto chunk_valid = [&](int64_t m) -> int {
    const int64_t rem = sg.t1 - (sg.t0 + m * C);
    return rem < C ? static_cast<int>(rem) : C;
  };

  float beta_reg = 0.f;  // beta of the next chunk to be scanned (threads < 64)
  if (tid < C && sg.t0 + tid < sg.t1 && kda_guard((sg.t0 + tid) * H + h, 1, a.T * H, a.err))
    beta_reg = a.beta[(sg.t0 + tid) * H + h];

  // ---- initial state, transposed into TMEM: S^T[j][c] = S_init[c][j] (worker warps)
  if (warp < kWarps) {
    const int j = 32 * quad + lane;
    const float* src = nullptr;  // buffer src_buf (src_n floats) at offset src_off
    const float* src_buf = nullptr;
    int64_t src_off = 0, src_n = 0;
    if (MODE == kModeReplay) {
      if (sg.index == 0) {
        src_buf = a.S0;
        src_off = (static_cast<int64_t>(sg.seq) * H + h) * DIO * DIO;
        src_n = static_cast<int64_t>(a.N) * H * DIO * DIO;
      } else {
        src_buf = a.entry_state;
        src_off = (static_cast<int64_t>(seg_id) * H + h) * D * D;
        src_n = static_cast<int64_t>(a.plan.capacity) * H * D * D;
      }
      if (src_buf) src = src_buf + src_off;
    }
    const int lds = (MODE == kModeReplay && sg.index == 0) ? DIO : D;  // row stride of src
#pragma unroll
    for (int cc = 0; cc < 32; cc += 16) {
      uint32_t r[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int c = 32 * part + cc + x;
        r[x] = __float_as_uint(
            src && c < lds && j < lds && kda_guard(src_off + c * lds + j, 1, src_n, a.err)
                ? src[c * lds + j]
                : 0.f);
      }
      tmem_st16(tmem_addr(tmem, 32 * quad, kColS + 32 * part + cc), r);
      if (kSum) {  // S_M = I
#pragma unroll
        for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(32 * part + cc + x == j ? 1.f : 0.f);
        tmem_st16(tmem_addr(tmem, 32 * quad, cSM + 32 * part + cc), r);
      }
    }
    tmem_wait_st();
  }

  ChunkRegs cr;
  float* sPC = reinterpret_cast<float*>(sm + kPC);
  // Decay scan of chunk m: raw q, k, log_alpha (TMA) -> registers (cr), the
  // strip anchors, the per-channel factors (sPC, e^{g_last} by parity) and
  // beta (sBeta).  Touches no operand buffer, so it can run while the tensor
  // core still reads the previous chunk's operands.  Starts the TMA of chunk
  // m+1's raw q, k, log_alpha once chunk m's are in registers.
  auto scan_chunk = [&](int64_t m) {
    const int valid = chunk_valid(m);
    if (!mbar_wait(bar_qkl, static_cast<uint32_t>(m & 1))) flag_timeout();
    float2 g[4][2];
    {
      float2 run01 = make_float2(0.f, 0.f), run23 = make_float2(0.f, 0.f);
      const bool full = valid == C;  // warp-uniform: no token of the chunk is past the end
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = r0 + i;
        const bool ok = full || r < valid;
        float2 la01, la23;
        if (FUSED) {  // gate logits, bf16
          float gf[4];
          unpack4(*reinterpret_cast<const uint2*>(sm + kRawL + sw128_offset(C, r, 8 * lane)), gf);
          la01 = make_float2(gate_log_alpha_fast(gf[0]), gate_log_alpha_fast(gf[1]));
          la23 = make_float2(gate_log_alpha_fast(gf[2]), gate_log_alpha_fast(gf[3]));
        } else {
          const float4 l4 =
              *reinterpret_cast<const float4*>(sm + kRawL + sw128_offset(C, r, 16 * lane));
          la01 = make_float2(clamp_log_alpha(l4.x), clamp_log_alpha(l4.y));
          la23 = make_float2(clamp_log_alpha(l4.z), clamp_log_alpha(l4.w));
        }
        if (ok) {
          run01 = add2(run01, la01);
          run23 = add2(run23, la23);
        }
        g[i][0] = run01;
        g[i][1] = run23;
        cr.kraw[i] = ok ? *reinterpret_cast<const uint2*>(sm + kRawK + sw128_offset(C, r, 8 * lane))
                        : make_uint2(0u, 0u);
        cr.qraw[i] = (kOut && ok)
                         ? *reinterpret_cast<const uint2*>(sm + kRawQ + sw128_offset(C, r, 8 * lane))
                         : make_uint2(0u, 0u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_raw);  // this warp is done with the raw tiles
      *reinterpret_cast<float4*>(sTot + warp * 128 + 4 * lane) =
          make_float4(run01.x, run01.y, run23.x, run23.y);
    }
    if (tid < C) sBeta[tid] = beta_reg;
    worker_sync();
    if (warp < 4) {
      // Across the 16 warps, lane = channel: the totals become exclusive
      // prefixes in place (added in warp order, as a serial scan would), the
      // anchors g_15, g_47, g_63 are the prefixes after warps 3, 11, 15, and
      // the per-channel factors follow from them.
      const int ch = 32 * warp + lane;
      float acc = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float t = sTot[w * 128 + ch];
        sTot[w * 128 + ch] = acc;
        acc += t;
        if (w == 3) a0 = acc;
        if (w == 11) a1 = acc;
      }
      sG0[ch] = a0;
      sG1[ch] = a1;
      sEGl[(m & 1) * 128 + ch] = __expf(acc);
      sPC[0 * 128 + ch] = __expf(a0);
      sPC[1 * 128 + ch] = __expf(a1);
      sPC[2 * 128 + ch] = __expf(acc - a0);
      sPC[3 * 128 + ch] = __expf(acc - a1);
      sPC[4 * 128 + ch] = __expf(a1 - a0);
    }
    if (tid < C) {
      const int64_t t = sg.t0 + (m + 1) * C + tid;
      beta_reg = t < sg.t1 && kda_guard(t * H + h, 1, a.T * H, a.err) ? a.beta[t * H + h] : 0.f;
    }
    worker_sync();
    {
      // g - G = (within-warp prefix) + (exclusive prefix of the earlier warps - G)
      const float4 off = *reinterpret_cast<const float4*>(sTot + warp * 128 + 4 * lane);
      const float4 gA = *reinterpret_cast<const float4*>((strip ? sG1 : sG0) + 4 * lane);
      const float2 d01 = sub2(lo2(off), lo2(gA)), d23 = sub2(hi2(off), hi2(gA));
      if (DUMP && dump_unit && m == a.dump_chunk) {  // g = within-warp prefix + earlier warps
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (kda_guard(kDumpG + (r0 + i) * 128 + 4 * lane, 4, kDumpFloats, a.err))
            *reinterpret_cast<float4*>(a.dump + kDumpG + (r0 + i) * 128 + 4 * lane) = make_float4(
                g[i][0].x + off.x, g[i][0].y + off.y, g[i][1].x + off.z, g[i][1].y + off.w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x01 = add2(g[i][0], d01), x23 = add2(g[i][1], d23);
        cr.e[i][0] = make_float2(__expf(x01.x), __expf(x01.y));  // in [e^-80, e^80]
        cr.e[i][1] = make_float2(__expf(x23.x), __expf(x23.y));
      }
    }
  };

  // Operand build of the scanned chunk: strip operands (bf16) and k e^g
  // (tf32) into SMEM, made visible to the tensor core: replay stores k e^g
  // [token][channel] (the B operand of P^T = S^T (k e^g)^T), summary
  // transposed (the A operand of W^T = (k e^g)^T T^T).  Reads cr and sPC
  // (written by scan_chunk, separated from here by a barrier).
  auto build_chunk = [&]() {
    unsigned char* Aop = R;           // bf16 [128][128]: strip s -> rows 64 s + (q: 0 | k: 32) + rr
    unsigned char* Bop = R + 32768;   // bf16 [96][128]: keys 0..31 (strip-0 anchor) | keys 0..63
    const float4 eg4 = *reinterpret_cast<const float4*>(sPC + (strip ? 1 : 0) * 128 + 4 * lane);
    const float4 e104 = *reinterpret_cast<const float4*>(sPC + 4 * 128 + 4 * lane);
    const float2 eG01 = lo2(eg4), eG23 = hi2(eg4), e1001 = lo2(e104), e1023 = hi2(e104);
    float kgT[4][4];                  // [channel x][token i] of k e^g (summary)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + i, rr = r & 31;
      float2 kf01, kf23, qf01, qf23;
      unpack4x2(cr.kraw[i], kf01, kf23);
      unpack4x2(cr.qraw[i], qf01, qf23);
      const float2 e01 = cr.e[i][0], e23 = cr.e[i][1];
      const float2 qt01 = mul2(qf01, e01), qt23 = mul2(qf23, e23);
      const float2 kt01 = mul2(kf01, e01), kt23 = mul2(kf23, e23);
      const float2 kh01 = mul2(kf01, rcp2(e01)), kh23 = mul2(kf23, rcp2(e23));
      const float2 kg01 = mul2(kt01, eG01), kg23 = mul2(kt23, eG23);
      kgT[0][i] = kg01.x; kgT[1][i] = kg01.y; kgT[2][i] = kg23.x; kgT[3][i] = kg23.y;
      if (kP) *reinterpret_cast<uint4*>(KG + sw128_offset(C, r, 16 * lane)) = pack4x2_tf32(kg01, kg23);
      *reinterpret_cast<uint2*>(Aop + sw128_offset(128, 64 * strip + rr, 8 * lane)) =
          pack4x2_bf16(qt01, qt23);
      *reinterpret_cast<uint2*>(Aop + sw128_offset(128, 64 * strip + 32 + rr, 8 * lane)) =
          pack4x2_bf16(kt01, kt23);
      if (strip == 0) {
        *reinterpret_cast<uint2*>(Bop + sw128_offset(96, r, 8 * lane)) = pack4x2_bf16(kh01, kh23);
        *reinterpret_cast<uint2*>(Bop + sw128_offset(96, 32 + r, 8 * lane)) =
            pack4x2_bf16(mul2(kh01, e1001), mul2(kh23, e1023));
      } else {
        *reinterpret_cast<uint2*>(Bop + sw128_offset(96, 32 + r, 8 * lane)) = pack4x2_bf16(kh01, kh23);
      }
    }
    if (!kP) {
      uint4 kv[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) kv[x] = pack4_tf32(kgT[x]);
      st_transposed4(KG, lane, r0, kv);
    }
    fence_proxy_async_smem();
  };

  // O^T of chunk m (TMEM) -> out, bf16.  Lanes = value channels, columns =
  // tokens; neighbouring lanes swap one value so each store writes a bf16 pair.
  auto write_out = [&](int64_t m) {
    const int valid = chunk_valid(m);
    const int64_t c0 = sg.t0 + m * C;
    const int j = 32 * quad + lane;
    uint32_t ov[16];
    tmem_ld16(tmem_addr(tmem, 32 * quad, kColO + 16 * part), ov);
    tmem_wait_ld();
    const bool odd = lane & 1;
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      const float v0 = __uint_as_float(ov[2 * y]), v1 = __uint_as_float(ov[2 * y + 1]);
      const float send = odd ? v0 : v1;
      const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
      const int t = 16 * part + 2 * y + (odd ? 1 : 0);
      const float lo = odd ? recv : v0, hi = odd ? v1 : recv;
      if (t < valid && j < DIO &&
          kda_guard(((c0 + t) * H + h) * DIO + (j & ~1), 2, a.T * H * DIO, a.err))
        *reinterpret_cast<uint32_t*>(a.out + ((c0 + t) * H + h) * DIO + (j & ~1)) = pack_bf16x2(lo, hi);
    }
  };

  // S^T (TMEM) -> buf[off + c * ld + j] = S[c][j] (row = key channel), f32, in a
  // buffer of n floats; worker warps.  Rows and columns below lim of the state
  // in TMEM columns col..
  auto store_state = [&](float* buf, int64_t off, int64_t n, int64_t ld, uint32_t col, int lim) {
    const int j = 32 * quad + lane;
#pragma unroll
    for (int cc = 0; cc < 32; cc += 16) {
      uint32_t sv[16];
      tmem_ld16(tmem_addr(tmem, 32 * quad, col + 32 * part + cc), sv);
      tmem_wait_ld();
      if (j < lim && 32 * part + cc < lim) {
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int64_t e = off + (32 * part + cc + x) * ld + j;
          if (kda_guard(e, 1, n, a.err)) buf[e] = __uint_as_float(sv[x]);
        }
      }
    }
  };
  // Phase F on one state: decay the columns of S^T (TMEM columns cs..) by
  // e^{g_last} of chunk n, round U^T (columns cu..) to tf32 in place.
  // Replay, warps 2..15: -P^T rounded to tf32 in place.  A warp reaches the
  // TMEM lanes of its quadrant (warp mod 4); the 4 blocks of 16 columns go
  // round-robin over that quadrant's warps (4, 8, 12 + q for q = 0, 1; q, 4,
  // 8, 12 + q for q = 2, 3).
  auto round_neg_p = [&]() {
    const int first = quad < 2 ? 4 + quad : quad, cnt = quad < 2 ? 3 : 4;
#pragma unroll 1
    for (int c = (warp - first) >> 2; c < 4; c += cnt) {
      const uint32_t ta = tmem_addr(tmem, 32 * quad, cP + 16 * c);
      uint32_t pv[16];
      tmem_ld16(ta, pv);
      tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 16; ++x) pv[x] = f32_to_tf32_rn(-__uint_as_float(pv[x]));
      tmem_st16(ta, pv);
      tmem_wait_st();
    }
  };
  // Replay: q e^g = q e^{g - G} e^G of this warp's tokens, [token][channel]
  // tf32 into KG (the B operand of O^T = S^T (q e^g)^T)
  auto write_qeg = [&]() {
    const float4 eg4 = *reinterpret_cast<const float4*>(sPC + (strip ? 1 : 0) * 128 + 4 * lane);
    const float2 eG01 = lo2(eg4), eG23 = hi2(eg4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 qf01, qf23;
      unpack4x2(cr.qraw[i], qf01, qf23);
      const float2 f01 = mul2(mul2(qf01, cr.e[i][0]), eG01), f23 = mul2(mul2(qf23, cr.e[i][1]), eG23);
      // fp32 as is: the tensor core reads it as tf32 by truncation, which on
      // this output-only operand costs well under the rounding budget
      *reinterpret_cast<float4*>(KG + sw128_offset(C, r0 + i, 16 * lane)) =
          make_float4(f01.x, f01.y, f23.x, f23.y);
    }
  };
  auto decay_round = [&](uint32_t cs, uint32_t cu, int64_t n) {
    const float* gl = sEGl + (n & 1) * 128 + 32 * part;
#pragma unroll
    for (int cc = 0; cc < 32; cc += 16) {
      const uint32_t ta = tmem_addr(tmem, 32 * quad, cs + 32 * part + cc);
      uint32_t sv[16];
      tmem_ld16(ta, sv);
      float4 gv[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) gv[y] = *reinterpret_cast<const float4*>(gl + cc + 4 * y);
      tmem_wait_ld();
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float2 a = mul2(make_float2(__uint_as_float(sv[4 * y]), __uint_as_float(sv[4 * y + 1])),
                              lo2(gv[y]));
        const float2 b = mul2(make_float2(__uint_as_float(sv[4 * y + 2]), __uint_as_float(sv[4 * y + 3])),
                              hi2(gv[y]));
        sv[4 * y] = __float_as_uint(a.x); sv[4 * y + 1] = __float_as_uint(a.y);
        sv[4 * y + 2] = __float_as_uint(b.x); sv[4 * y + 3] = __float_as_uint(b.y);
      }
      tmem_st16(ta, sv);
    }
    const uint32_t tu = tmem_addr(tmem, 32 * quad, cu + 16 * part);
    uint32_t uv[16];
    tmem_ld16(tu, uv);
    tmem_wait_ld();
#pragma unroll
    for (int x = 0; x < 16; ++x) uv[x] = f32_to_tf32_rn(__uint_as_float(uv[x]));
    tmem_st16(tu, uv);
    tmem_wait_st();
  };
  // ================= control warps: issue the MMA groups once their operands are ready.
  // Issuing a tcgen05.mma costs the issuing thread ~100 cycles, far more than
  // the tensor pipe needs for these shapes, so the independent MMA chains of
  // each group are issued by two threads in parallel (issuer 0 and 1, lane 0
  // of the two control warps).  Each issuer commits its own chain.
  auto control = [&](int who) {
    // K-major SW128 operand, 8-row groups 1024 B apart: K step j of a
    // [blocks][rows][128 B] tile starts at block j / 4, byte (j % 4) * 32.  The
    // start address is the descriptor's low field, so a step is an add to the
    // tile's base descriptor.
    auto kmaj = [](uint64_t base_desc, int j, uint32_t block_bytes) {
      return base_desc + (((j >> 2) * block_bytes + (j & 3) * 32) >> 4);
    };
    auto kdesc = [](const void* p) { return smem_desc_sw128(smem_u32(p), 16, 1024); };
    if (who == 1 && n_chunks > 0) {
      issue_qkl(sg.t0);
      issue_v(sg.t0);
    }
    if (tin && who == 0 && n_chunks > 0 && !*s_abort)
      bulk_prefetch_l2(t_rec(0), static_cast<uint32_t>(kTChunkBytes));
    for (int64_t n = 0; n < n_chunks; ++n) {
      if (who == 1) {  // raw q, k, log_alpha of chunk n read by every worker: stream in n+1
        if (*s_abort) break;
        if (!mbar_wait(bar_raw, static_cast<uint32_t>(n & 1))) { flag_timeout(); break; }
        if (n + 1 < n_chunks) issue_qkl(sg.t0 + (n + 1) * C);
      }
      if constexpr (kP) {  // replay: groups 0 | P, 1, 3
        const uint32_t id64 = make_idesc(kFmtTF32, 128, 64, false, false);
        // group 0: strip products (issuer 0); P^T = S^T (k e^g)^T once the
        // previous chunk's state update has completed (issuer 1)
        bool ready = mbar_wait(bar_ready + 0, static_cast<uint32_t>(n & 1));
        if (ready && who == 1 && n > 0)
          ready = mbar_wait(bar_done + 3, static_cast<uint32_t>((n - 1) & 1));
        if (!ready) flag_timeout();
        tc_fence_after();
        bool go = ready && !*s_abort;
        if (who == 0) {
          if (go) {
            const uint32_t id = make_idesc(kFmtBF16, 128, 96, false, false);
            const uint64_t a0 = kdesc(R), b0 = kdesc(R + 32768);
#pragma unroll 2
            for (int j = 0; j < D / 16; ++j)
              mma_f16_ss(tmem + cA, kmaj(a0, j, 128 * 128), kmaj(b0, j, 96 * 128), id, j > 0);
          }
          mma_commit(bar_done + 0);
          // TIN: chunk n's T record into R (the strip A operand) once the
          // strip MMA has read it; chunk n+1's record on its way into L2
          if (tin && go) {
            if (mbar_wait(bar_done + 0, static_cast<uint32_t>(n & 1))) {
              mbar_arrive_expect_tx(bar_t, static_cast<uint32_t>(kTChunkBytes));
              bulk_load(R, t_rec(n), static_cast<uint32_t>(kTChunkBytes), bar_t);
              if (n + 1 < n_chunks)
                bulk_prefetch_l2(t_rec(n + 1), static_cast<uint32_t>(kTChunkBytes));
            } else {
              flag_timeout();
            }
          }
        } else {
          if (go) {
            const uint64_t kg = kdesc(KG);
#pragma unroll 2
            for (int j = 0; j < D / 8; ++j)
              mma_tf32_ts(tmem + cP, tmem + kColS + 8 * j, kmaj(kg, j, 64 * 128), id64, j > 0);
          }
          mma_commit(bar_donep);
        }
        if (*s_abort) break;
        // group 1: O^T = S^T (q e^g)^T (issuer 0); U^T = V^T T^T (bf16 hi + lo)
        // + (-P^T) T^T (issuer 1)
        ready = mbar_wait(bar_ready + 1, static_cast<uint32_t>(n & 1));
        if (!ready) flag_timeout();
        tc_fence_after();
        go = ready && !*s_abort;
        if (who == 0) {
          if (go) {
            const uint64_t qg = kdesc(KG);
#pragma unroll 2
            for (int j = 0; j < D / 8; ++j)
              mma_tf32_ts(tmem + kColO, tmem + kColS + 8 * j, kmaj(qg, j, 64 * 128), id64, j > 0);
          }
          mma_commit(bar_done + 1);
        } else {
          bool ok = go;
          if (ok && !mbar_wait(bar_v, static_cast<uint32_t>(n & 1))) { flag_timeout(); ok = false; }
          if (tin && ok && !mbar_wait(bar_t, static_cast<uint32_t>(n & 1))) {
            flag_timeout();
            ok = false;
          }
          tc_fence_after();
          if (ok) {
            const uint32_t idu = make_idesc(kFmtBF16, 128, 64, true, false);
            const uint64_t vv = smem_desc_sw128(smem_u32(sm + kRawV), 64 * 128, 1024);
            const uint64_t th = kdesc(R + kRTh), tl = kdesc(R + kRTl);
#pragma unroll 2
            for (int j = 0; j < 2 * (C / 16); ++j) {  // hi half (j < 4), then lo half
              const int jj = j & 3;
              mma_f16_ss(tmem + cU, vv + ((jj * 2048) >> 4), (j < 4 ? th : tl) + ((jj * 32) >> 4),
                         idu, j > 0);
            }
            const uint64_t tt = kdesc(R + kRT);
#pragma unroll 2
            for (int j = 0; j < C / 8; ++j)
              mma_tf32_ts(tmem + cU, tmem + cP + 8 * j, kmaj(tt, j, 64 * 128), id64, 1);
          }
          mma_commit(bar_done + 1);
          // raw v of chunk n consumed once group 1 has completed: stream in n+1
          if (n + 1 < n_chunks) {
            if (mbar_wait(bar_done + 1, static_cast<uint32_t>(n & 1))) issue_v(sg.t0 + (n + 1) * C);
            else flag_timeout();
          }
        }
        if (*s_abort) break;
        // group 3: S^T += U^T K' (issuer 0); O^T += U^T A_qk^T (issuer 1)
        ready = mbar_wait(bar_ready + 3, static_cast<uint32_t>(n & 1));
        if (!ready) flag_timeout();
        tc_fence_after();
        go = ready && !*s_abort;
        if (go && who == 0) {
          const uint32_t ids = make_idesc(kFmtTF32, 128, 128, false, false);
          const uint64_t kp = kdesc(KP);
#pragma unroll 2
          for (int j = 0; j < C / 8; ++j)
            mma_tf32_ts(tmem + kColS, tmem + cU + 8 * j, kmaj(kp, j, 128 * 128), ids, 1);
        }
        if (go && who == 1) {
          const uint64_t aq = kdesc(R + kRAqk);
#pragma unroll 2
          for (int j = 0; j < C / 8; ++j)
            mma_tf32_ts(tmem + kColO, tmem + cU + 8 * j, kmaj(aq, j, 64 * 128), id64, 1);
        }
        mma_commit(bar_done + 3);
        if (*s_abort) break;
      } else {  // summary: groups 0..3
        for (int g = 0; g < 4; ++g) {
          if (*s_abort) break;
          const bool ready = mbar_wait(bar_ready + g, static_cast<uint32_t>(n & 1));
          if (!ready) flag_timeout();
          tc_fence_after();
          const bool go = ready && !*s_abort;
          if (g == 0) {
            if (who == 0) {  // strip products (bf16)
              if (go) {
                const uint32_t id = make_idesc(kFmtBF16, 128, 96, false, false);
                const uint64_t a0 = kdesc(R), b0 = kdesc(R + 32768);
  #pragma unroll 4
                for (int j = 0; j < D / 16; ++j)
                  mma_f16_ss(tmem + cA, kmaj(a0, j, 128 * 128), kmaj(b0, j, 96 * 128), id, j > 0);
              }
              mma_commit(bar_done + 0);
            }
          } else if (g == 1) {
            if (who == 0) {  // W^T = (k e^g)^T T^T (tf32)
              if (go && t_ok) {  // T of chunk n kept for the replay of this segment
                bulk_store(t_rec(n), R, static_cast<uint32_t>(kTChunkBytes));
                bulk_commit();
              }
              if (go) {
                const uint32_t idw = make_idesc(kFmtTF32, 128, 64, false, false);
                const uint64_t kg = kdesc(KG), tt = kdesc(R + kRT);
  #pragma unroll 4
                for (int j = 0; j < C / 8; ++j)
                  mma_tf32_ss(tmem + cW, kmaj(kg, j, 128 * 128), kmaj(tt, j, 64 * 128), idw, j > 0);
              }
            } else {  // U~^T = V^T T^T (bf16 hi + lo), once raw v has landed
              bool ok = go;
              if (ok && !mbar_wait(bar_v, static_cast<uint32_t>(n & 1))) { flag_timeout(); ok = false; }
              tc_fence_after();
              if (ok) {
                const uint32_t idu = make_idesc(kFmtBF16, 128, 64, true, false);
                const uint64_t vv = smem_desc_sw128(smem_u32(sm + kRawV), 64 * 128, 1024);
                const uint64_t th = kdesc(R + kRTh), tl = kdesc(R + kRTl);
  #pragma unroll 4
                for (int j = 0; j < 2 * (C / 16); ++j) {  // hi half (j < 4), then lo half
                  const int jj = j & 3;
                  mma_f16_ss(tmem + cU, vv + ((jj * 2048) >> 4), (j < 4 ? th : tl) + ((jj * 32) >> 4),
                             idu, j > 0);
                }
              }
            }
            mma_commit(bar_done + 1);
            // raw v of chunk n consumed once group 1 has completed: stream in n+1
            if (who == 1 && n + 1 < n_chunks) {
              if (mbar_wait(bar_done + 1, static_cast<uint32_t>(n & 1))) issue_v(sg.t0 + (n + 1) * C);
              else flag_timeout();
            }
          } else if (g == 2) {
            // the T record has left R before this group commits (the workers
            // overwrite R once group 2 has completed)
            if (t_ok && who == 0) bulk_wait_read();
            const uint32_t id = make_idesc(kFmtTF32, 128, 64, false, false);
            if (go && who == 0) {  // U^T -= S^T W^T (KG holds -W)
              const uint64_t wm = kdesc(KG);
  #pragma unroll 4
              for (int j = 0; j < D / 8; ++j)
                mma_tf32_ts(tmem + cU, tmem + kColS + 8 * j, kmaj(wm, j, 64 * 128), id, 1);
            }
            if (go && who == 1) {  // U_M^T = -S_M^T W^T (no values)
              const uint64_t wm = kdesc(KG);
  #pragma unroll 4
              for (int j = 0; j < D / 8; ++j)
                mma_tf32_ts(tmem + cUM, tmem + cSM + 8 * j, kmaj(wm, j, 64 * 128), id, j > 0);
            }
            mma_commit(bar_done + 2);
          } else {
            if (go && who == 1) {  // S_M^T += U_M^T K'
              const uint32_t ids = make_idesc(kFmtTF32, 128, 128, false, false);
              const uint64_t kp = kdesc(KP);
  #pragma unroll 4
              for (int j = 0; j < C / 8; ++j)
                mma_tf32_ts(tmem + cSM, tmem + cUM + 8 * j, kmaj(kp, j, 128 * 128), ids, 1);
            }
            if (go && who == 0) {  // S^T += U^T K'
              const uint32_t ids = make_idesc(kFmtTF32, 128, 128, false, false);
              const uint64_t kp = kdesc(KP);
  #pragma unroll 4
              for (int j = 0; j < C / 8; ++j)
                mma_tf32_ts(tmem + kColS, tmem + cU + 8 * j, kmaj(kp, j, 128 * 128), ids, 1);
            }
            mma_commit(bar_done + 3);
          }
        }
      }
      if (*s_abort) break;
    }
    if (kSum && t_ok && who == 0) bulk_wait();  // the T records are written before exit
  };

  if (warp >= kWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp < kWarps + 2 && lane == 0) control(warp - kWarps);
    __syncwarp();
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kWorkerRegs));
    // checkpoints: the segment's first token within its sequence, read once
    // here (a global load at the end of every chunk would sit on the chain);
    // negative: the unit writes none
    int32_t ck_seg_off = -1;
    if (CKPT && kda_guard(sg.first, 1, a.plan.capacity, a.err) && kda_guard(sg.seq, 1, a.N, a.err))
      ck_seg_off = static_cast<int32_t>(sg.t0 - a.plan.segs[sg.first].t0);
    if (n_chunks > 0) {
      scan_chunk(0);
      worker_sync();
      if (FUSED) l2norm8_bf16(cr.kraw, cr.qraw, lane);  // q, k of the warp's 4 tokens
      build_chunk();
      signal_ready(0);  // strip operands of chunk 0
    }
    for (int64_t n = 0; n < n_chunks; ++n) {
      if (*s_abort) break;

      // ---- A: strip products (bf16) -> TMEM  ||  out of chunk n-1
      if (kOut && n > 0) write_out(n - 1);
      wait_done_sync(0, n);
      if (*s_abort) break;
      const bool dump_chunk = DUMP && dump_unit && n == a.dump_chunk;
      if (dump_chunk) store_state(a.dump, kDumpS, kDumpFloats, 128, kColS, D);  // S at the chunk's start

      // ---- B: strip read-out, UT transform, T to SMEM (TIN: T arrives by
      //      TMA, and only the query rows are read out)
      if (!tin || !(quad & 1)) {
        // row L = 32 quad + lane of the strip products: strip s = quad / 2,
        // query rows (A_qk) for even quad, key rows (A_kk) for odd; token r.
        const int s = quad >> 1, is_k = quad & 1;
        const int r = 32 * s + lane;
        const int nk = s ? 16 : 8;  // keys handled by this warp: [i0, i0 + nk)
        const int i0 = part * nk;
        uint32_t v[16];
        const uint32_t ta = tmem_addr(tmem, 32 * quad, cA + (s ? 32u : 0u) + i0);
        if (s) tmem_ld16(ta, v); else tmem_ld8(ta, v);
        tmem_wait_ld();
        const float b = sBeta[r];
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          if (g4 * 4 >= nk) break;
          float f[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int i = i0 + 4 * g4 + x;
            const float val = __uint_as_float(v[4 * g4 + x]);
            f[x] = is_k ? ((i < r) ? b * val : 0.f) : ((i <= r) ? val : 0.f);
          }
          const int i = i0 + 4 * g4;
          if (is_k) {
            *reinterpret_cast<float4*>(sAkk + r * kLdA + i) = make_float4(f[0], f[1], f[2], f[3]);
            if (s == 1 && i < 32) {  // transposed copy of A_(10) for the inverse
              float* a10t = reinterpret_cast<float*>(KP);
#pragma unroll
              for (int x = 0; x < 4; ++x) a10t[(i + x) * 32 + lane] = f[x];
            }
          }
          else if (kOut)
            *reinterpret_cast<float4*>(R + kRAqk + sw128_offset(C, r, 4 * i)) =
                make_float4(f[0], f[1], f[2], f[3]);  // output-only: read truncated
        }
        if (s == 0) {  // strip-0 rows have no keys >= 32
          const int iz = 32 + 8 * part;
          if (is_k) {
            *reinterpret_cast<float4*>(sAkk + r * kLdA + iz) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(sAkk + r * kLdA + iz + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (kOut) {
            *reinterpret_cast<uint4*>(R + kRAqk + sw128_offset(C, r, 4 * iz)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(R + kRAqk + sw128_offset(C, r, 4 * iz + 16)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (dump_chunk) {  // A_kk (beta applied) and A_qk, before the inverse overwrites A_kk
        worker_sync();
        for (int e = tid; e < C * C; e += kWorkers) {
          const int r = e >> 6, i = e & 63;
          if (kda_guard(kDumpAqk + e, 1, kDumpFloats, a.err)) {
            a.dump[kDumpAkk + e] = sAkk[r * kLdA + i];
            a.dump[kDumpAqk + e] =
                *reinterpret_cast<const float*>(R + kRAqk + sw128_offset(C, r, 4 * i));
          }
        }
        worker_sync();
      }
      if (tin) {
        // once P^T has landed: -P^T rounded to tf32 in TMEM (one 16-column
        // block per warp) and q e^g into KG (P^T's B operand is consumed)
        if (warp == 0 && !mbar_wait(bar_donep, static_cast<uint32_t>(n & 1))) flag_timeout();
        worker_sync();
        tc_fence_after();
        {
          const uint32_t ta = tmem_addr(tmem, 32 * quad, cP + 16 * part);
          uint32_t pv[16];
          tmem_ld16(ta, pv);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) pv[x] = f32_to_tf32_rn(-__uint_as_float(pv[x]));
          tmem_st16(ta, pv);
          tmem_wait_st();
        }
        write_qeg();
      } else {
      // The inverse reads only the key rows (odd lane quadrants, A_kk); its
      // first step runs on warps 0 and 1.  Those nine warps meet here; the
      // query-row warps (A_qk) join at the inverse's next barrier, so their
      // longer read-out overlaps the diagonal blocks.
      if (warp == 0 || (warp & 1)) asm volatile("bar.sync 2, 288;" ::: "memory");
      ut_front(sAkk, reinterpret_cast<float*>(R + kRXs), R, tid);
      // replay: once P^T has landed, -P^T rounded to tf32 in TMEM (warps 2..15,
      // which are free here) and q e^g into KG (P^T's B operand is consumed);
      // warps 0 and 1 write their q e^g after the transform
      if (kP && warp >= 2) {
        if (warp == 2 && !mbar_wait(bar_donep, static_cast<uint32_t>(n & 1))) flag_timeout();
        asm volatile("bar.sync 3, 448;" ::: "memory");  // warps 2..15
        tc_fence_after();
        round_neg_p();
        write_qeg();
      }
      worker_sync();
      ut_back(sAkk, reinterpret_cast<float*>(R + kRXs), reinterpret_cast<const float*>(KP), sBeta,
              R, tid);
      if (kP && warp < 2) {
        if (!mbar_wait(bar_donep, static_cast<uint32_t>(n & 1))) flag_timeout();
        tc_fence_after();
        write_qeg();
      }
      if (kP) worker_sync();  // K' and the next scan start after the transform's critical step
      }
      if (dump_chunk) {  // T (its tf32 operand copy)
        for (int e = tid; e < C * C; e += kWorkers) {
          const int r = e >> 6, i = e & 63;
          if (kda_guard(kDumpT + e, 1, kDumpFloats, a.err))
            a.dump[kDumpT + e] = *reinterpret_cast<const float*>(R + kRT + sw128_offset(C, r, 4 * i));
        }
      }
      signal_ready(1);  // T, V (and k e^g | -P^T, q e^g) ready for group 1

      // ---- C: W^T = (k e^g)^T T^T (tf32), U~^T = V^T T^T (bf16 hi + lo)  ||  K' to SMEM
      {
        // K' = k e^{g_last - g} = k e^{G - g} e^{g_last - G}, transposed [c][t]
        const float4 gl4 = *reinterpret_cast<const float4*>(sPC + (strip ? 3 : 2) * 128 + 4 * lane);
        const float2 gl01 = lo2(gl4), gl23 = hi2(gl4);
        float kp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 kf01, kf23;
          unpack4x2(cr.kraw[i], kf01, kf23);
          const float2 p01 = mul2(mul2(kf01, rcp2(cr.e[i][0])), gl01);
          const float2 p23 = mul2(mul2(kf23, rcp2(cr.e[i][1])), gl23);
          kp[0][i] = p01.x; kp[1][i] = p01.y; kp[2][i] = p23.x; kp[3][i] = p23.y;
        }
        uint4 kv[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) kv[x] = pack4_tf32(kp[x]);
        if (kOut) st_rows4(KP, lane, r0, kv);
        else st_transposed4(KP, lane, r0, kv);
      }
      if (kP && n + 1 < n_chunks) scan_chunk(n + 1);  // registers + small tables only
      wait_done_sync(1, n);
      if (*s_abort) break;
      if (dump_chunk) {  // U = T (V - k e^g S), before its tf32 rounding: U^T lanes = value channels
        const int j = 32 * quad + lane;
        uint32_t uv[16];
        tmem_ld16(tmem_addr(tmem, 32 * quad, cU + 16 * part), uv);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          if (kda_guard(kDumpU + (16 * part + x) * 128 + j, 1, kDumpFloats, a.err))
            a.dump[kDumpU + (16 * part + x) * 128 + j] = __uint_as_float(uv[x]);
      }

      if (!kP) {  // summary: phases D and E

      // ---- D: -W (from W^T in TMEM, lane = key channel) to SMEM
      {
        const int c = 32 * quad + lane;
        uint32_t w[16];
        tmem_ld16(tmem_addr(tmem, 32 * quad, cW + 16 * part), w);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          *reinterpret_cast<uint32_t*>(KG + sw128_offset(C, 16 * part + x, 4 * c)) =
              f32_to_tf32_rn(-__uint_as_float(w[x]));
      }
      signal_ready(2);  // -W ready

      // ---- E: U^T -= S^T W^T (A = S^T in TMEM)  ||  scan of chunk n+1
      if (n + 1 < n_chunks) scan_chunk(n + 1);  // registers + small tables only
      wait_done_sync(2, n);
      if (*s_abort) break;
      }

      // ---- F: decay the columns of S^T by e^{g_last}; round U^T to tf32
      //      (summary: both S_B^T and S_M^T, U_B^T and U_M^T)
      decay_round(kColS, cU, n);
      if (kSum) decay_round(cSM, cUM, n);
      signal_ready(3);  // S^T decayed, U^T rounded, A_qk and K' in SMEM

      // ---- G: O^T += U^T A_qk^T ; S^T += U^T K'  (A = U^T)  ||  chunk n+1 operand build
      if (n + 1 < n_chunks) {
        // fused preparation: L2-normalise chunk n+1's q and k here, beside the
        // state MMAs, rather than in its decay scan, which sits on the path
        // of phase C
        if (FUSED) l2norm8_bf16(cr.kraw, cr.qraw, lane);
        build_chunk();  // chunk n+1 operands into freed buffers
        signal_ready(0);
      }
      wait_done_sync(3, n);
      if (CKPT && ck_seg_off >= 0) {  // the state after this chunk, if the sequence has a checkpoint here
        // tokens of the sequence up to this chunk's end (< 2^31: TMA coordinates are 32-bit)
        const int32_t ci = static_cast<int32_t>(a.plan.ckpt_interval);
        const int32_t pos = ck_seg_off + static_cast<int32_t>(n) * C + chunk_valid(n);
        if (pos % ci == 0) {
          const int64_t slot = a.plan.ckpt_base[sg.seq] + pos / ci - 1;
          if (slot < a.plan.ckpt_max) {  // 8 columns at a time: few live registers mid-loop
            const int64_t ck_off = (slot * H + h) * DIO * DIO;
            const int64_t ck_n = a.plan.ckpt_max * H * DIO * DIO;
            float* dst = a.ckpt + ck_off;
            const int j = 32 * quad + lane;
#pragma unroll 1
            for (int cc = 0; cc < 32; cc += 8) {
              uint32_t sv[16];
              tmem_ld8(tmem_addr(tmem, 32 * quad, kColS + 32 * part + cc), sv);
              tmem_wait_ld();
              if (j < DIO && 32 * part + cc < DIO) {
#pragma unroll
                for (int x = 0; x < 8; ++x)
                  if (kda_guard(ck_off + (32 * part + cc + x) * DIO + j, 1, ck_n, a.err))
                    dst[(32 * part + cc + x) * DIO + j] = __uint_as_float(sv[x]);
              }
            }
          }
        }
      }
    }

    if (kOut && n_chunks > 0 && !*s_abort) write_out(n_chunks - 1);

    // ---- the segment's final state (S^T in TMEM) to global memory
    if (!*s_abort) {
      if (MODE == kModeReplay) {
        if (last && a.S_final)
          store_state(a.S_final, (static_cast<int64_t>(sg.seq) * H + h) * DIO * DIO,
                      static_cast<int64_t>(a.N) * H * DIO * DIO, DIO, kColS, DIO);
        else if (a.plan.first_replayed && !last && sg.index == 0 && a.entry_state)
          // the first pass's replay of segment 0: the entry state of segment 1
          store_state(a.entry_state, (static_cast<int64_t>(seg_id + 1) * H + h) * D * D,
                      static_cast<int64_t>(a.plan.capacity) * H * D * D, D, kColS, D);
      } else {  // the increment | transition record, rows of 2 D floats
        const int64_t off = (static_cast<int64_t>(seg_id) * H + h) * D * (2 * D);
        const int64_t n_it = static_cast<int64_t>(a.plan.capacity) * H * D * (2 * D);
        store_state(a.incr_trans, off, n_it, 2 * D, kColS, D);
        store_state(a.incr_trans, off + D, n_it, 2 * D, cSM, D);
      }
    }
  }  // worker warps
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarps) tmem_dealloc(tmem, kTmemCols);
}

// CKPT (replay only): write the state checkpoints the plan asks for; a separate
// instantiation, so the plain replay keeps its register budget.
// DUMP (replay only): also write the intermediates of one chunk of one unit
// (a.dump); a separate instantiation with extra barriers, for debugging.
template <int MODE, bool FUSED, bool CKPT, bool DUMP = false>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ TcMaps maps, PrefillArgs a) {
  int32_t seg_id;
  Segment sg;
  int h;
  if (!unit_of(a, seg_id, sg, h)) return;
  prefill_tc_body<MODE, FUSED, CKPT, DUMP>(maps, a, seg_id, sg, h);
}

// First pass of a split prefill, one launch: every segment but the last one
// of its sequence is summarised, except that with first_replayed (uniform
// batches) the first segment of every sequence is replayed from S0 instead,
// writing its outputs and the entry state of segment 1.
template <bool FUSED, bool CKPT>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pass1_kernel(const __grid_constant__ TcMaps maps, PrefillArgs a) {
  int32_t seg_id;
  Segment sg;
  int h;
  if (!unit_of(a, seg_id, sg, h)) return;
  if (a.plan.first_replayed && sg.index == 0)
    prefill_tc_body<kModeReplay, FUSED, CKPT, false>(maps, a, seg_id, sg, h);
  else
    prefill_tc_body<kModeSummary, FUSED, false, false>(maps, a, seg_id, sg, h);
}

// Second pass of a split prefill: the segments left are replayed from their
// entry states.  Every one but the last of its sequence was summarised in
// the first pass, and with the T records kept it loads them (TIN).
template <bool FUSED, bool CKPT>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pass2_kernel(const __grid_constant__ TcMaps maps, PrefillArgs a) {
  int32_t seg_id;
  Segment sg;
  int h;
  if (!unit_of(a, seg_id, sg, h)) return;
  prefill_tc_body<kModeReplay, FUSED, CKPT, false, true>(maps, a, seg_id, sg, h);
}

// ---- host side: TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [T][H][128] tensor viewed as 3-D (channel, head, token); box = box_c channels
// x 1 head x 64 tokens, 128-byte swizzle.  Rows past T read as zero.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int64_t T,
              int H, int dch, uint32_t box_c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(dch), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(dch) * esize,
                                 static_cast<cuuint64_t>(H) * dch * esize};
  const cuuint32_t box[3] = {box_c, 1, static_cast<cuuint32_t>(C)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The kernel a launch runs: one mode (PASS 0), or a split prefill's first
// (1) or second (2) pass.
template <int MODE, bool FUSED, bool CKPT, bool DUMP, int PASS>
struct KernelOf {
  static constexpr auto fn = prefill_tc_kernel<MODE, FUSED, CKPT, DUMP>;
};
template <int MODE, bool FUSED, bool CKPT, bool DUMP>
struct KernelOf<MODE, FUSED, CKPT, DUMP, 1> {
  static constexpr auto fn = prefill_pass1_kernel<FUSED, CKPT>;
};
template <int MODE, bool FUSED, bool CKPT, bool DUMP>
struct KernelOf<MODE, FUSED, CKPT, DUMP, 2> {
  static constexpr auto fn = prefill_pass2_kernel<FUSED, CKPT>;
};

template <int MODE, bool FUSED, bool CKPT, bool DUMP = false, int PASS = 0>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t s, const char* name) {
  constexpr auto kern = KernelOf<MODE, FUSED, CKPT, DUMP, PASS>::fn;
  if (a.T > 0x7fffffffLL) return cudaErrorInvalidValue;  // TMA coordinates are 32-bit
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  if (a.T > 0) {
    const int dch = a.dv;  // 64: the boxes past channel 63 read as zeros
    const bool ok =
        make_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, dch, 64) &&
        make_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, dch, 64) &&
        make_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, dch, 64) &&
        (FUSED ? make_map(&maps.la, a.gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, dch, 64)
               : make_map(&maps.la, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H, dch,
                          32));
    if (!ok) return cudaErrorInvalidValue;
  }
  // The register split inside the kernel assumes the launch allocation; a
  // build that allocates fewer registers per thread is not launched (its
  // setmaxnreg.inc could never be satisfied).
  static int launch_regs = -1;
  if (launch_regs < 0) {
    cudaFuncAttributes fa;
    const cudaError_t ea = cudaFuncGetAttributes(&fa, kern);
    if (ea != cudaSuccess) return ea;
    launch_regs = fa.numRegs;
  }
  if (static_cast<uint32_t>(launch_regs) < kLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.plan.capacity) * a.H;  // (segment, head) blocks
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<uint32_t>(units), 1, 1);
  prof_begin(s, name);
  kern<<<grid, kThreads, kSmemBytes, s>>>(maps, a);
  prof_end(s, name);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_pass1(const PrefillArgs& a, cudaStream_t s) {
  if (a.ckpt)
    return a.fused ? launch_tc<kModeReplay, true, true, false, 1>(a, s, "kda_prefill_pass1")
                   : launch_tc<kModeReplay, false, true, false, 1>(a, s, "kda_prefill_pass1");
  return a.fused ? launch_tc<kModeReplay, true, false, false, 1>(a, s, "kda_prefill_pass1")
                 : launch_tc<kModeReplay, false, false, false, 1>(a, s, "kda_prefill_pass1");
}

cudaError_t launch_prefill_pass2(const PrefillArgs& a, cudaStream_t s) {
  if (a.ckpt)
    return a.fused ? launch_tc<kModeReplay, true, true, false, 2>(a, s, "kda_prefill_replay")
                   : launch_tc<kModeReplay, false, true, false, 2>(a, s, "kda_prefill_replay");
  return a.fused ? launch_tc<kModeReplay, true, false, false, 2>(a, s, "kda_prefill_replay")
                 : launch_tc<kModeReplay, false, false, false, 2>(a, s, "kda_prefill_replay");
}

cudaError_t launch_prefill_replay_dump(const PrefillArgs& a, cudaStream_t s) {
  return launch_tc<kModeReplay, false, false, true>(a, s, "kda_prefill_replay_dump");
}

cudaError_t launch_prefill_replay(const PrefillArgs& a, cudaStream_t s) {
  if (a.ckpt)
    return a.fused ? launch_tc<kModeReplay, true, true>(a, s, "kda_prefill_replay")
                   : launch_tc<kModeReplay, false, true>(a, s, "kda_prefill_replay");
  return a.fused ? launch_tc<kModeReplay, true, false>(a, s, "kda_prefill_replay")
                 : launch_tc<kModeReplay, false, false>(a, s, "kda_prefill_replay");
}

}  // namespace kda
