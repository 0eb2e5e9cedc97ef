// Chunk-parallel prefill on the tcgen05 tensor cores (dk = dv = 128).
//
// One CTA per unit = (segment, head[, column kind]) walks the segment's
// 64-token chunks in order.  The state is kept TRANSPOSED in tensor memory
// (S^T: lane = value channel j, column = key channel c, fp32) for the whole
// segment and is itself the A operand of the MMAs that read it, so it never
// leaves the SM between chunks.  Per chunk (tokens r, i of the chunk, g the
// within-chunk cumulative clamped log-decay per key channel):
//
//   strip products (bf16):  A_qk[r,i] = sum_c q_rc k_ic e^{g_rc - g_ic}  (i <= r)
//                           A_kk[r,i] = beta_r sum_c k_rc k_ic e^{g_rc - g_ic}  (i < r)
//   UT transform (fp32):    T = (I + A_kk)^{-1} Diag(beta)
//   WY products (tf32/bf16): W^T = (k e^g)^T T^T,   U~^T = V^T T^T
//   hand-off (tf32):        U^T = U~^T - S^T W^T
//                           O^T = S^T (q e^g)^T + U^T A_qk^T        -> out
//                           S^T <- S^T Diag(e^{g_last}) + U^T (k e^{g_last - g})
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
// the state path is tf32 rounded to nearest; accumulation is fp32.
//
// Phases of one chunk (256 threads, one MMA-issuing thread):
//   1 decay scan + operand build (registers -> swizzled SMEM)   all warps
//   2 strip MMA -> TMEM                                          thread 0
//   3 strip read-out, UT transform                               all warps
// (tf32 operands are always laid out K-major: the key-side factors k e^g and
// K' are written transposed, [key channel][token].)
//   4 W^T, U~^T MMAs                                             thread 0
//   5 -W and q e^g to SMEM                                       all warps
//   6 U^T -= S^T W^T ; O^T = S^T (q e^g)^T                       thread 0
//   7 S^T column decay, U^T rounding, K' to SMEM                 all warps
//   8 O^T += U^T A_qk^T ; S^T += U^T K'                          thread 0
//   9 O^T -> out                                                 all warps
// Raw q, k, log_alpha of the next chunk stream in by TMA from phase 1 on,
// v from phase 4 on.
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
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

// TMEM column map (fp32 columns; 128 lanes)
constexpr uint32_t kColS = 0;     // S^T          128 columns
constexpr uint32_t kColA = 128;   // strip products 96 columns
constexpr uint32_t kColW = 256;   // W^T           64 columns (lane = key channel)
constexpr uint32_t kColU = 320;   // U^T           64 columns (lane = value channel)
constexpr uint32_t kColO = 384;   // O^T           64 columns

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kRawQ = 0;                 // bf16 [64][128] sw128 (2 blocks)
constexpr uint32_t kRawK = kRawQ + 16384;
constexpr uint32_t kRawV = kRawK + 16384;
constexpr uint32_t kRawL = kRawV + 16384;     // f32 [64][128] sw128 (4 blocks)
constexpr uint32_t kR = kRawL + 32768;        // phase-dependent operand region
//   phase 1-2: strip A operand bf16 [128][128] at R, strip B operand [96][128] at R+32768
//   phase 3-4: A_qk tf32 [64][64] at R, T tf32 at R+16384, T_hi/T_lo bf16 at R+32768/+40960,
//              A_kk scratch f32 [64][kLdA] at R+49152, T' scratch f32 at R+49152+kScr
//   phase 5-8: A_qk at R, q e^g tf32 [64][128] at R+16384
//   phase 9:   output tile bf16 [64][128] (plain rows) at R+16384
constexpr uint32_t kLdA = 68;                 // padded row stride (floats) of the scratch matrices
constexpr uint32_t kScr = C * kLdA * 4;       // 17408
constexpr uint32_t kRBytes = 49152 + 2 * kScr;
// k e^g (transposed, [128 c][64 t]) -> -W ([64 t][128 c]) -> K' (transposed), all tf32 K-major
constexpr uint32_t kKG = kR + ((kRBytes + 1023) / 1024) * 1024;
constexpr uint32_t kMisc = kKG + 32768;
// misc (floats): warp totals [8][128], G0 [128], G1 [128], g_last [128], e^{g_last} [128],
// e^{G1 - G0} [128], beta [64]
constexpr uint32_t kTot = kMisc;
constexpr uint32_t kG0 = kTot + 8 * 128 * 4;
constexpr uint32_t kG1 = kG0 + 512;
constexpr uint32_t kGl = kG1 + 512;
constexpr uint32_t kEGl = kGl + 512;
constexpr uint32_t kE10 = kEGl + 512;
constexpr uint32_t kBeta = kE10 + 512;
constexpr uint32_t kBars = kBeta + 256;       // 3 mbarriers + TMEM slot
constexpr uint32_t kSmemBytes = kBars + 64 + 1024;  // + alignment slack

struct TcMaps {
  CUtensorMap q, k, v, la;
};

enum : int { kModeSummary = 0, kModeReplay = 1 };

// Read 4 consecutive f32 (channels 4l..4l+3) of row r from a sw128 f32 tile.
__device__ __forceinline__ float4 ld_f32x4(const unsigned char* tile, int r, int l) {
  return *reinterpret_cast<const float4*>(tile + sw128_offset(C, r, 16 * l));
}
// Read 4 consecutive bf16 of row r (channels 4l..4l+3) from a sw128 bf16 tile.
__device__ __forceinline__ uint2 ld_bf16x4(const unsigned char* tile, int r, int l) {
  return *reinterpret_cast<const uint2*>(tile + sw128_offset(C, r, 8 * l));
}
__device__ __forceinline__ void unpack4(uint2 u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}
// Store 4 bf16 (channels 4l..) into row `row` of a sw128 bf16 tile with `rows` rows.
__device__ __forceinline__ void st_bf16x4(unsigned char* tile, uint32_t rows, int row, int l,
                                          const float (&f)[4]) {
  uint2 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  *reinterpret_cast<uint2*>(tile + sw128_offset(rows, row, 8 * l)) = u;
}
// Store 4 tf32 (channels 4l..) into row `row` of a sw128 32-bit tile with `rows` rows.
__device__ __forceinline__ void st_tf32x4(unsigned char* tile, uint32_t rows, int row, int l,
                                          const float (&f)[4]) {
  uint4 u;
  u.x = f32_to_tf32_rn(f[0]);
  u.y = f32_to_tf32_rn(f[1]);
  u.z = f32_to_tf32_rn(f[2]);
  u.w = f32_to_tf32_rn(f[3]);
  *reinterpret_cast<uint4*>(tile + sw128_offset(rows, row, 16 * l)) = u;
}

// T' = (I + A)^{-1} for a strictly lower-triangular 64 x 64 matrix A (fp32,
// row stride kLdA).  The four 16 x 16 diagonal blocks are inverted by forward
// substitution (one thread per column), then block rows are combined:
// T'_ab = -T'_aa sum_{b <= c < a} A_ac T'_cb.  sT must be zero on entry.
__device__ void unit_lower_inverse(const float* __restrict__ sA, float* __restrict__ sT, int tid) {
  if (tid < 64) {
    const int b = tid >> 4, j = tid & 15;
    const float* Ab = sA + (16 * b) * kLdA + 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) s += Ab[r * kLdA + i] * x[i];
      if (r > j) x[r] = -s;
    }
    float* Tb = sT + (16 * b) * kLdA + 16 * b;
#pragma unroll
    for (int r = 0; r < 16; ++r) Tb[r * kLdA + j] = x[r];
  }
  __syncthreads();
  const int rr = tid >> 4, cc = tid & 15;
  for (int a = 1; a < 4; ++a) {
    float xv[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      if (b >= a) break;
      float s = 0.f;
      for (int c = b; c < a; ++c) {
        const float* Arow = sA + (16 * a + rr) * kLdA + 16 * c;
        const float* Tcol = sT + (16 * c) * kLdA + 16 * b + cc;
#pragma unroll
        for (int i = 0; i < 16; ++i) s += Arow[i] * Tcol[i * kLdA];
      }
      xv[b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 3; ++b)
      if (b < a) sT[(16 * a + rr) * kLdA + 16 * b + cc] = xv[b];
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      if (b >= a) break;
      const float* Drow = sT + (16 * a + rr) * kLdA + 16 * a;
      const float* Xcol = sT + (16 * a) * kLdA + 16 * b + cc;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) s += Drow[i] * Xcol[i * kLdA];
      xv[b] = -s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 3; ++b)
      if (b < a) sT[(16 * a + rr) * kLdA + 16 * b + cc] = xv[b];
    __syncthreads();
  }
}

// Store 8 consecutive tokens (t0..t0+7) of channel c as tf32 into a K-major
// [128 channels][64 tokens] tile (the transposed layout of key-side factors).
__device__ __forceinline__ void st_tf32_col8(unsigned char* tile, int c, int t0, const float (&v)[8]) {
  uint4 u0, u1;
  u0.x = f32_to_tf32_rn(v[0]); u0.y = f32_to_tf32_rn(v[1]);
  u0.z = f32_to_tf32_rn(v[2]); u0.w = f32_to_tf32_rn(v[3]);
  u1.x = f32_to_tf32_rn(v[4]); u1.y = f32_to_tf32_rn(v[5]);
  u1.z = f32_to_tf32_rn(v[6]); u1.w = f32_to_tf32_rn(v[7]);
  *reinterpret_cast<uint4*>(tile + sw128_offset(D, c, 4 * t0)) = u0;
  *reinterpret_cast<uint4*>(tile + sw128_offset(D, c, 4 * t0 + 16)) = u1;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ TcMaps maps, PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t seg_id = blockIdx.x;
  const int h = blockIdx.y;
  if (seg_id >= *a.plan.n_segs) return;
  const Segment sg = a.plan.segs[seg_id];
  const bool last = sg.index + 1 == sg.count;
  if (MODE == kModeSummary && last) return;
  // summary units: z = 0 accumulates the increment B (values, zero start),
  // z = 1 the transition M (no values, identity start)
  const bool ident = MODE == kModeSummary && blockIdx.z == 1;
  const bool has_v = !ident;
  constexpr bool kOut = MODE == kModeReplay;
  const int H = a.H;

  uint64_t* bar_qkl = reinterpret_cast<uint64_t*>(sm + kBars);
  uint64_t* bar_v = bar_qkl + 1;
  uint64_t* bar_mma = bar_qkl + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_qkl + 3);
  int* s_abort = reinterpret_cast<int*>(tslot + 1);
  float* sTot = reinterpret_cast<float*>(sm + kTot);
  float* sG0 = reinterpret_cast<float*>(sm + kG0);
  float* sG1 = reinterpret_cast<float*>(sm + kG1);
  float* sGl = reinterpret_cast<float*>(sm + kGl);
  float* sEGl = reinterpret_cast<float*>(sm + kEGl);
  float* sBeta = reinterpret_cast<float*>(sm + kBeta);
  unsigned char* R = sm + kR;
  unsigned char* KG = sm + kKG;
  float* sAkk = reinterpret_cast<float*>(R + 49152);
  float* sTp = reinterpret_cast<float*>(R + 49152 + kScr);

  const int64_t n_chunks = (sg.t1 - sg.t0 + C - 1) / C;
  const uint32_t qkl_bytes = kOut ? 65536u : 49152u;

  if (tid == 0) {
    mbar_init(bar_qkl, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
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
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_3d(sm + kRawL + 8192 * b, &maps.la, 32 * b, h, t, bar_qkl);
  };
  auto issue_v = [&](int64_t c0) {
    mbar_arrive_expect_tx(bar_v, 16384u);
    const int32_t t = static_cast<int32_t>(c0);
    tma_load_3d(sm + kRawV, &maps.v, 0, h, t, bar_v);
    tma_load_3d(sm + kRawV + 8192, &maps.v, 64, h, t, bar_v);
  };
  if (tid == 0 && n_chunks > 0) {
    issue_qkl(sg.t0);
    if (has_v) issue_v(sg.t0);
  }
  float beta_next = 0.f;
  if (tid < C && sg.t0 + tid < sg.t1) beta_next = a.beta[(sg.t0 + tid) * H + h];

  // ---- initial state, transposed into TMEM: S^T[j][c] = S_init[c][j]
  const int quad = warp & 3, half = warp >> 2;
  {
    const int j = 32 * quad + lane;
    const float* src = nullptr;
    if (MODE == kModeReplay) {
      if (sg.index == 0)
        src = a.S0 ? a.S0 + (static_cast<int64_t>(sg.seq) * H + h) * D * D : nullptr;
      else
        src = a.entry_state + (static_cast<int64_t>(seg_id) * H + h) * D * D;
    }
#pragma unroll
    for (int cc = 0; cc < 64; cc += 16) {
      uint32_t r[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int c = 64 * half + cc + x;
        float v = 0.f;
        if (ident) v = (c == j) ? 1.f : 0.f;
        else if (src) v = src[c * D + j];
        r[x] = __float_as_uint(v);
      }
      tmem_st16(tmem_addr(tmem, 32 * quad, kColS + 64 * half + cc), r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint32_t mma_par = 0;
  // bounded wait on the MMA barrier by every thread; false = give up
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(bar_mma, mma_par);
    mma_par ^= 1u;
    if (!ok) { atomicOr(a.err, kDevErrTimeout); *s_abort = 1; }
    tc_fence_after();
    return ok;
  };

  const int r0 = 8 * warp;      // this thread's tokens r0 .. r0+7 (phases 1, 5, 7)
  const int strip = warp >> 2;  // their 32-token strip
  for (int64_t ci = 0; ci < n_chunks; ++ci) {
    const int64_t c0 = sg.t0 + ci * C;
    const int valid = (sg.t1 - c0) < C ? static_cast<int>(sg.t1 - c0) : C;

    // ================= phase 1: decay scan and operand build
    {
      const bool ok = mbar_wait(bar_qkl, static_cast<uint32_t>(ci & 1));
      if (!ok) { atomicOr(a.err, kDevErrTimeout); *s_abort = 1; }
    }
    float e[8][4];   // e^{g - G_strip}, kept for phases 5 and 7
    uint2 kraw[8], qraw[8];
    {
      float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + i;
        const float4 l4 = ld_f32x4(sm + kRawL, r, lane);
        const bool ok = r < valid;
        run[0] += ok ? clamp_log_alpha(l4.x) : 0.f;
        run[1] += ok ? clamp_log_alpha(l4.y) : 0.f;
        run[2] += ok ? clamp_log_alpha(l4.z) : 0.f;
        run[3] += ok ? clamp_log_alpha(l4.w) : 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) e[i][x] = run[x];  // local prefix for now
        kraw[i] = ok ? ld_bf16x4(sm + kRawK, r, lane) : make_uint2(0u, 0u);
        qraw[i] = (kOut && ok) ? ld_bf16x4(sm + kRawQ, r, lane) : make_uint2(0u, 0u);
      }
      *reinterpret_cast<float4*>(sTot + warp * 128 + 4 * lane) =
          make_float4(run[0], run[1], run[2], run[3]);
    }
    if (tid < C) sBeta[tid] = beta_next;
    __syncthreads();
    if (*s_abort) break;
    // raw q, k, log_alpha are in registers now: stream in the next chunk's
    if (tid == 0 && ci + 1 < n_chunks) issue_qkl(c0 + C);
    {
      float off[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = 0; w < warp; ++w) {
        const float4 t4 = *reinterpret_cast<const float4*>(sTot + w * 128 + 4 * lane);
        off[0] += t4.x; off[1] += t4.y; off[2] += t4.z; off[3] += t4.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int x = 0; x < 4; ++x) e[i][x] += off[x];  // now g
      // anchors: token 15 (warp 1), token 47 (warp 5), last token 63 (warp 7)
      float* dst = warp == 1 ? sG0 : warp == 5 ? sG1 : warp == 7 ? sGl : nullptr;
      if (dst)
        *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(e[7][0], e[7][1], e[7][2], e[7][3]);
      if (warp == 7)
        *reinterpret_cast<float4*>(sEGl + 4 * lane) =
            make_float4(__expf(e[7][0]), __expf(e[7][1]), __expf(e[7][2]), __expf(e[7][3]));
    }
    __syncthreads();
    float eG[4], eglG[4], e10[4];  // e^{G}, e^{g_last - G}, e^{G1 - G0} (own channels)
    {
      const float4 g0 = *reinterpret_cast<const float4*>(sG0 + 4 * lane);
      const float4 g1 = *reinterpret_cast<const float4*>(sG1 + 4 * lane);
      const float4 gl = *reinterpret_cast<const float4*>(sGl + 4 * lane);
      const float G[4] = {strip ? g1.x : g0.x, strip ? g1.y : g0.y, strip ? g1.z : g0.z,
                          strip ? g1.w : g0.w};
      const float GL[4] = {gl.x, gl.y, gl.z, gl.w};
      const float D10[4] = {g1.x - g0.x, g1.y - g0.y, g1.z - g0.z, g1.w - g0.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        eG[x] = __expf(G[x]);
        eglG[x] = __expf(GL[x] - G[x]);
        e10[x] = __expf(D10[x]);
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i][x] = __expf(e[i][x] - G[x]);  // within [e^-80, e^80]
      }
    }
    {
      unsigned char* Aop = R;           // bf16 [128 rows][128]: strip s -> rows 64s + (q | k) * 32 + rr
      unsigned char* Bop = R + 32768;   // bf16 [96 rows][128]: keys of strip 0 | keys of strip 1
      float kgT[4][8];                  // k e^g for the transposed store
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + i, rr = r & 31;
        float kf[4], qf[4], qt[4], kt[4], kh[4];
        unpack4(kraw[i], kf);
        unpack4(qraw[i], qf);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float inv = __frcp_rn(e[i][x]);
          qt[x] = qf[x] * e[i][x];
          kt[x] = kf[x] * e[i][x];
          kh[x] = kf[x] * inv;
          kgT[x][i] = kt[x] * eG[x];
        }
        if (kOut) st_bf16x4(Aop, 128, 64 * strip + rr, lane, qt);
        st_bf16x4(Aop, 128, 64 * strip + 32 + rr, lane, kt);
        if (strip == 0) {
          st_bf16x4(Bop, 96, r, lane, kh);
          float kh1[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) kh1[x] = kh[x] * e10[x];
          st_bf16x4(Bop, 96, 32 + r, lane, kh1);
        } else {
          st_bf16x4(Bop, 96, 32 + r, lane, kh);
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) st_tf32_col8(KG, 4 * lane + x, r0, kgT[x]);
      if (!kOut) {  // summary units have no queries: keep the strip rows finite
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) st_bf16x4(Aop, 128, 64 * strip + ((r0 + i) & 31), lane, z);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ================= phase 2: strip products (bf16) -> TMEM
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = make_idesc(kFmtBF16, 128, 96, false, false);
      const uint32_t a0 = smem_u32(R), b0 = smem_u32(R + 32768);
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const uint64_t ad = smem_desc_sw128(a0 + (j >> 2) * (128 * 128) + (j & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc_sw128(b0 + (j >> 2) * (96 * 128) + (j & 3) * 32, 16, 1024);
        mma_f16_ss(tmem + kColA, ad, bd, id, j > 0);
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_mma();
    __syncthreads();
    if (*s_abort) break;

    // ================= phase 3: strip read-out, UT transform
    for (int i = tid; i < C * static_cast<int>(kLdA); i += kThreads) sTp[i] = 0.f;
    if (warp < 4) {
      // row L = 32 warp + lane of the strip product: strip s = warp / 2,
      // warp even = query rows (A_qk), odd = key rows (A_kk); token r.
      const int s = warp >> 1, is_k = warp & 1;
      const int r = 32 * s + lane;
      uint32_t v[64];
#pragma unroll
      for (int i = 32; i < 64; ++i) v[i] = 0u;
      const uint32_t col0 = kColA + (s ? 32u : 0u);
      const uint32_t ta = tmem_addr(tmem, 32 * warp, col0);
      tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
      tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
      if (s) {
        tmem_ld16(ta + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
        tmem_ld16(ta + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
      }
      tmem_wait_ld();
      const int nkeys = s ? 64 : 32;
      if (!is_k) {
        if (kOut) {  // A_qk row r, tf32, K-major [r][i], zero above the diagonal
#pragma unroll
          for (int l4 = 0; l4 < 16; ++l4) {
            float f[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int i = 4 * l4 + x;
              f[x] = (i <= r && i < nkeys) ? __uint_as_float(v[i]) : 0.f;
            }
            st_tf32x4(R, C, r, l4, f);
          }
        }
      } else {
        const float b = sBeta[r];
        float* row = sAkk + r * kLdA;
#pragma unroll
        for (int l4 = 0; l4 < 16; ++l4) {
          float f[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * l4 + x;
            f[x] = (i < r && i < nkeys) ? b * __uint_as_float(v[i]) : 0.f;
          }
          *reinterpret_cast<float4*>(row + 4 * l4) = make_float4(f[0], f[1], f[2], f[3]);
        }
      }
    }
    __syncthreads();
    unit_lower_inverse(sAkk, sTp, tid);
    {
      // T = T' Diag(beta): row r = tid / 4, columns 16 (tid % 4) .. +16
      const int r = tid >> 2, i0 = 16 * (tid & 3);
      unsigned char* Tt = R + 16384;    // tf32 [64][64]
      unsigned char* Th = R + 32768;    // bf16 [64][64] high part
      unsigned char* Tl = R + 40960;    // bf16 low part
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float f[4], hi[4], lo[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int i = i0 + 4 * q4 + x;
          f[x] = sTp[r * kLdA + i] * sBeta[i];
          hi[x] = __bfloat162float(__float2bfloat16_rn(f[x]));
          lo[x] = f[x] - hi[x];
        }
        const int l4 = (i0 >> 2) + q4;
        st_tf32x4(Tt, C, r, l4, f);
        st_bf16x4(Th, C, r, l4, hi);
        st_bf16x4(Tl, C, r, l4, lo);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ================= phase 4: W^T = (k e^g)^T T^T (tf32), U~^T = V^T T^T (bf16 hi + lo)
    if (tid == 0) {
      bool ok = true;
      if (has_v) {
        ok = mbar_wait(bar_v, static_cast<uint32_t>(ci & 1));
        if (!ok) { atomicOr(a.err, kDevErrTimeout); *s_abort = 1; }
      }
      tc_fence_after();
      if (ok) {
        const uint32_t idw = make_idesc(kFmtTF32, 128, 64, false, false);
        const uint32_t kg = smem_u32(KG), tt = smem_u32(R + 16384);
#pragma unroll
        for (int j = 0; j < C / 8; ++j) {
          const uint64_t ad = smem_desc_sw128(kg + (j >> 2) * (128 * 128) + (j & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(tt + (j >> 2) * (64 * 128) + (j & 3) * 32, 16, 1024);
          mma_tf32_ss(tmem + kColW, ad, bd, idw, j > 0);
        }
        if (has_v) {
          const uint32_t idu = make_idesc(kFmtBF16, 128, 64, true, false);
          const uint32_t vv = smem_u32(sm + kRawV);
          const uint32_t th = smem_u32(R + 32768), tl = smem_u32(R + 40960);
#pragma unroll
          for (int j = 0; j < C / 16; ++j) {
            const uint64_t ad = smem_desc_sw128(vv + j * 2048, 64 * 128, 1024);
            mma_f16_ss(tmem + kColU, ad, smem_desc_sw128(th + j * 32, 16, 1024), idu, j > 0);
          }
#pragma unroll
          for (int j = 0; j < C / 16; ++j) {
            const uint64_t ad = smem_desc_sw128(vv + j * 2048, 64 * 128, 1024);
            mma_f16_ss(tmem + kColU, ad, smem_desc_sw128(tl + j * 32, 16, 1024), idu, 1);
          }
        }
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_mma();
    __syncthreads();
    if (*s_abort) break;
    if (tid == 0 && has_v && ci + 1 < n_chunks) issue_v(c0 + C);

    // ================= phase 5: -W (from W^T in TMEM) and q e^g to SMEM
    {
      // W^T: lane = key channel c, column = token; this warp: tokens 32 half .. +32
      const int c = 32 * quad + lane;
#pragma unroll
      for (int t16 = 0; t16 < 32; t16 += 16) {
        uint32_t w[16];
        tmem_ld16(tmem_addr(tmem, 32 * quad, kColW + 32 * half + t16), w);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int r = 32 * half + t16 + x;
          *reinterpret_cast<uint32_t*>(KG + sw128_offset(C, r, 4 * c)) =
              f32_to_tf32_rn(-__uint_as_float(w[x]));
        }
      }
      if (kOut) {
        unsigned char* QG = R + 16384;  // tf32 [64 tokens][128]
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float qf[4], f[4];
          unpack4(qraw[i], qf);
#pragma unroll
          for (int x = 0; x < 4; ++x) f[x] = qf[x] * e[i][x] * eG[x];
          st_tf32x4(QG, C, r0 + i, lane, f);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ================= phase 6: U^T -= S^T W^T ; O^T = S^T (q e^g)^T   (A = S^T in TMEM)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = make_idesc(kFmtTF32, 128, 64, false, false);
      const uint32_t wm = smem_u32(KG), qg = smem_u32(R + 16384);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const uint64_t bd = smem_desc_sw128(wm + (j >> 2) * (64 * 128) + (j & 3) * 32, 16, 1024);
        mma_tf32_ts(tmem + kColU, tmem + kColS + 8 * j, bd, id, (has_v || j > 0) ? 1u : 0u);
      }
      if (kOut) {
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          const uint64_t bd = smem_desc_sw128(qg + (j >> 2) * (64 * 128) + (j & 3) * 32, 16, 1024);
          mma_tf32_ts(tmem + kColO, tmem + kColS + 8 * j, bd, id, j > 0);
        }
      }
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_mma();
    __syncthreads();
    if (*s_abort) break;

    // ================= phase 7: decay S^T columns, round U^T, K' to SMEM
    {
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) {
        const uint32_t ta = tmem_addr(tmem, 32 * quad, kColS + 64 * half + cc);
        uint32_t sv[16];
        tmem_ld16(ta, sv);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          sv[x] = __float_as_uint(__uint_as_float(sv[x]) * sEGl[64 * half + cc + x]);
        tmem_st16(ta, sv);
      }
#pragma unroll
      for (int cc = 0; cc < 32; cc += 16) {
        const uint32_t ta = tmem_addr(tmem, 32 * quad, kColU + 32 * half + cc);
        uint32_t uv[16];
        tmem_ld16(ta, uv);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x) uv[x] = f32_to_tf32_rn(__uint_as_float(uv[x]));
        tmem_st16(ta, uv);
      }
      tmem_wait_st();
      // K' = k e^{g_last - g} = k (e^{G - g}) e^{g_last - G}, transposed [c][t]
      float kp[4][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float kf[4];
        unpack4(kraw[i], kf);
#pragma unroll
        for (int x = 0; x < 4; ++x) kp[x][i] = kf[x] * __frcp_rn(e[i][x]) * eglG[x];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) st_tf32_col8(KG, 4 * lane + x, r0, kp[x]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ================= phase 8: O^T += U^T A_qk^T ; S^T += U^T K'   (A = U^T in TMEM)
    if (tid == 0) {
      tc_fence_after();
      if (kOut) {
        const uint32_t id = make_idesc(kFmtTF32, 128, 64, false, false);
        const uint32_t aq = smem_u32(R);
#pragma unroll
        for (int j = 0; j < C / 8; ++j) {
          const uint64_t bd = smem_desc_sw128(aq + (j >> 2) * (64 * 128) + (j & 3) * 32, 16, 1024);
          mma_tf32_ts(tmem + kColO, tmem + kColU + 8 * j, bd, id, 1);
        }
      }
      const uint32_t ids = make_idesc(kFmtTF32, 128, 128, false, false);
      const uint32_t kp = smem_u32(KG);
#pragma unroll
      for (int j = 0; j < C / 8; ++j) {
        const uint64_t bd = smem_desc_sw128(kp + (j >> 2) * (128 * 128) + (j & 3) * 32, 16, 1024);
        mma_tf32_ts(tmem + kColS, tmem + kColU + 8 * j, bd, ids, 1);
      }
      mma_commit(bar_mma);
    }
    if (tid < C) beta_next = (c0 + C + tid < sg.t1) ? a.beta[(c0 + C + tid) * H + h] : 0.f;
    __syncwarp();
    wait_mma();
    __syncthreads();
    if (*s_abort) break;

    // ================= phase 9: O^T -> out (bf16)
    if (kOut) {
      uint16_t* so = reinterpret_cast<uint16_t*>(R + 16384);  // [64 tokens][128] plain rows
      const int j = 32 * quad + lane;
#pragma unroll
      for (int t16 = 0; t16 < 32; t16 += 16) {
        uint32_t ov[16];
        tmem_ld16(tmem_addr(tmem, 32 * quad, kColO + 32 * half + t16), ov);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          so[(32 * half + t16 + x) * D + j] = f32_to_bf16(__uint_as_float(ov[x]));
      }
      __syncthreads();
      const int r = tid >> 2, qtr = tid & 3;  // row, 64-byte quarter
      if (r < valid) {
        const uint4* srcv = reinterpret_cast<const uint4*>(so + r * D + 32 * qtr);
        uint4* dstv = reinterpret_cast<uint4*>(a.out + ((c0 + r) * H + h) * D + 32 * qtr);
#pragma unroll
        for (int x = 0; x < 4; ++x) dstv[x] = srcv[x];
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // ---- the segment's final state (S^T in TMEM) to global memory
  if (!*s_abort) {
    float* dst = nullptr;
    int64_t ld = D;  // row stride of the destination (floats)
    if (MODE == kModeReplay) {
      if (last && a.S_final) dst = a.S_final + (static_cast<int64_t>(sg.seq) * H + h) * D * D;
    } else {
      ld = 2 * D;  // increment | transition record
      dst = a.incr_trans + (static_cast<int64_t>(seg_id) * H + h) * D * (2 * D) + (ident ? D : 0);
    }
    if (dst) {
      const int j = 32 * quad + lane;
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) {
        uint32_t sv[16];
        tmem_ld16(tmem_addr(tmem, 32 * quad, kColS + 64 * half + cc), sv);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x) dst[(64 * half + cc + x) * ld + j] = __uint_as_float(sv[x]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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
              int H, uint32_t box_c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esize,
                                 static_cast<cuuint64_t>(H) * D * esize};
  const cuuint32_t box[3] = {box_c, 1, static_cast<cuuint32_t>(C)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t s, const char* name) {
  if (a.T <= 0 || a.T > 0x7fffffffLL) {
    if (a.T > 0x7fffffffLL) return cudaErrorInvalidValue;
  }
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  if (a.T > 0) {
    const bool ok = make_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) &&
                    make_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) &&
                    make_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) &&
                    make_map(&maps.la, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H, 32);
    if (!ok) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  dim3 grid(a.plan.capacity, a.H, MODE == kModeSummary ? 2 : 1);
  prof_begin(s, name);
  prefill_tc_kernel<MODE><<<grid, kThreads, kSmemBytes, s>>>(maps, a);
  prof_end(s, name);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_summary_tc(const PrefillArgs& a, cudaStream_t s) {
  return launch_tc<kModeSummary>(a, s, "kda_prefill_summary");
}

cudaError_t launch_prefill_replay_tc(const PrefillArgs& a, cudaStream_t s) {
  return launch_tc<kModeReplay>(a, s, "kda_prefill_replay");
}

}  // namespace kda
