// Prefill schedule on the device, and the segment scan.
//
// The planner turns cu_seqlens (read on the GPU, so the host never waits)
// into a list of segments: each sequence is cut into pieces of
// `segment_tokens` tokens (a multiple of the 64-token chunk, so chunk
// boundaries stay aligned to the sequence start), or kept whole.
//
// Splitting follows the decomposition the pages describe for spreading one
// long sequence over many processors (meridianbulletin.com article, section
// "Parallelizing Sequential State Updates"; orkas.ai close read, section "The
// bill comes due in the serving stack"): a segment maps its entry state
// affinely, S_end = M S_in + B, where B is the segment run from a zero state
// and M the segment's transition.  The first pass computes (B_j, M_j) of
// every segment but each sequence's last; the scan below chains them,
// S_in(j+1) = M_j S_in(j) + B_j, and the second pass replays every segment
// from its exact entry state.  In a uniform batch the first pass replays
// segment 0 instead of summarising it (its exit state is S_in(1)), so the
// second pass replays segments 1 .. count - 1 only.
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ cu, int64_t T, int32_t N, int64_t L, Plan plan,
            int* err) {
  __shared__ int s_bad;
  __shared__ int32_t s_scan[kPlanThreads];
  __shared__ int32_t s_base;
  __shared__ int64_t s_cscan[kPlanThreads];  // checkpoint counts
  __shared__ int64_t s_cbase;
  const int tid = threadIdx.x;
  const int64_t CI = plan.ckpt_interval;
  if (tid == 0) {
    s_bad = 0; s_base = 0; s_cbase = 0;
    if (plan.n_order) plan.n_order[0] = plan.n_order[1] = 0;  // no units unless the plan completes
  }
  __syncthreads();

  // 1. validate cu_seqlens
  if (cu) {
    if (tid == 0 && kda_guard(N, 1, static_cast<int64_t>(N) + 1, err) &&
        (cu[0] != 0 || static_cast<int64_t>(cu[N]) != T))
      atomicOr(&s_bad, 1);
    for (int n = tid; n < N; n += kPlanThreads)
      if (kda_guard(n, 2, static_cast<int64_t>(N) + 1, err) && cu[n + 1] < cu[n]) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) { atomicOr(err, kDevErrCuSeqlens); *plan.n_segs = 0; }
    return;
  }
  const int64_t uni = N > 0 ? T / N : 0;

  // 2. segments per sequence, exclusive scan, emit
  for (int base = 0; base < N; base += kPlanThreads) {
    const int n = base + tid;
    int64_t t0 = 0, len = 0;
    int32_t cnt = 0;
    if (n < N && (!cu || kda_guard(n, 2, static_cast<int64_t>(N) + 1, err))) {
      t0 = cu ? cu[n] : uni * n;
      len = cu ? static_cast<int64_t>(cu[n + 1]) - cu[n] : uni;
      cnt = 1;
      if (L > 0 && len > L) cnt = static_cast<int32_t>((len + L - 1) / L);
    }
    const int64_t ccnt = (n < N && CI > 0) ? len / CI : 0;  // checkpoints of this sequence
    s_scan[tid] = cnt;
    s_cscan[tid] = ccnt;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {  // Hillis-Steele inclusive scans
      int32_t add = tid >= off ? s_scan[tid - off] : 0;
      int64_t cadd = tid >= off ? s_cscan[tid - off] : 0;
      __syncthreads();
      s_scan[tid] += add;
      s_cscan[tid] += cadd;
      __syncthreads();
    }
    if (n < N && CI > 0 && kda_guard(n, 1, N, err)) plan.ckpt_base[n] = s_cbase + s_cscan[tid] - ccnt;
    const int32_t first = s_base + s_scan[tid] - cnt;
    if (n < N) {
      for (int32_t j = 0; j < cnt; ++j) {
        const int32_t id = first + j;
        if (id >= plan.capacity) { atomicOr(&s_bad, 2); break; }
        Segment sg;
        sg.t0 = t0 + (L > 0 ? static_cast<int64_t>(j) * L : 0);
        sg.t1 = (j + 1 == cnt) ? t0 + len : sg.t0 + L;
        sg.seq = n;
        sg.index = j;
        sg.count = cnt;
        sg.first = first;
        if (kda_guard(id, 1, plan.capacity, err)) plan.segs[id] = sg;
      }
    }
    __syncthreads();
    if (tid == kPlanThreads - 1) { s_base += s_scan[tid]; s_cbase += s_cscan[tid]; }
    __syncthreads();
  }
  if (tid == 0 && CI > 0 && s_cbase > plan.ckpt_max) atomicOr(err, kDevErrCheckpoints);
  if (tid == 0) {
    if (s_bad) {
      atomicOr(err, kDevErrCapacity);
      *plan.n_segs = 0;
    } else {
      *plan.n_segs = s_base;
    }
  }

  // 3. launch orders, longest segment first.  The chunk kernels give each SM
  // the next (segment, head) unit as one frees, so starting the long units
  // first keeps the short ones (the last segment of each sequence, short
  // sequences) for the tail.  Counting sort on the chunk count (1024 buckets;
  // counts above 1023 share the top one), decreasing; the order inside a
  // bucket is whichever the atomics give, which changes only the schedule,
  // never a result.  The lists are those of Plan::order and Plan::order2
  // (kda_internal.h); unsplit, list 0 holds every segment.
  if (plan.order == nullptr) return;
  __syncthreads();
  if (s_bad) return;
  const int32_t ns = s_base;
  int32_t* s_count = s_scan;  // reused: [key]
  // sort key: the unit's modelled time in chunk-times (a second-pass replay
  // that loads its T records takes 0.77 of one per chunk)
  auto key_of = [&](int32_t id, int list) {
    const Segment& g = plan.segs[id];
    const int64_t chunks = (g.t1 - g.t0 + kChunk - 1) / kChunk;
    const bool loads_t = list == 1 && plan.t_records && g.index + 1 < g.count;
    const int64_t t = loads_t ? chunks * 77 / 100 : chunks;
    return static_cast<int>(t < kPlanThreads - 1 ? t : kPlanThreads - 1);
  };
  for (int list = 0; list < 2; ++list) {
    int32_t* out = list ? plan.order2 : plan.order;
    auto in_list = [&](int32_t id) {
      const Segment& g = plan.segs[id];
      if (L <= 0) return list == 0;  // unsplit: one pass over every segment
      if (plan.first_replayed) return list ? g.index >= 1 : (g.index == 0 || g.index + 1 < g.count);
      return list ? true : g.index + 1 < g.count;
    };
    s_count[tid] = 0;
    __syncthreads();
    for (int32_t id = tid; id < ns; id += kPlanThreads)
      if (kda_guard(id, 1, plan.capacity, err) && in_list(id)) atomicAdd(&s_count[key_of(id, list)], 1);
    __syncthreads();
    // first rank of key k = number of listed segments with a larger key: an
    // inclusive scan in decreasing key order (thread tid holds key
    // kPlanThreads - 1 - tid)
    const int my_key = kPlanThreads - 1 - tid;
    const int32_t my_count = s_count[my_key];
    __syncthreads();
    s_count[tid] = my_count;  // now indexed by position in decreasing-key order
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
      const int32_t add = tid >= off ? s_count[tid - off] : 0;
      __syncthreads();
      s_count[tid] += add;
      __syncthreads();
    }
    const int32_t first = s_count[tid] - my_count;
    if (tid == kPlanThreads - 1) plan.n_order[list] = s_count[tid];  // the list's length
    __syncthreads();
    s_count[my_key] = first;  // back to indexing by key: next free rank of that key
    __syncthreads();
    for (int32_t id = tid; id < ns; id += kPlanThreads) {
      if (!kda_guard(id, 1, plan.capacity, err) || !in_list(id)) continue;
      const int32_t rank = atomicAdd(&s_count[key_of(id, list)], 1);
      if (kda_guard(rank, 1, plan.capacity, err)) out[rank] = id;
    }
    __syncthreads();  // s_count is reused by the next list
  }
}

// Entry states of split sequences, S_in(j+1) = M_j S_in(j) + B_j, from S0 or,
// when the first pass replayed segment 0, from the S_in(1) it wrote: one CTA per
// (sequence, head, block of kScanCols state columns), sequential over the
// sequence's segments.  The whole M_j (D x D f32, from the summary records)
// is staged in shared memory by cp.async, the next segment's copy in flight
// while the current one is used.  The CTA's columns of S_in are kept
// transposed, so a thread reads 4 consecutive m of its M rows and of its
// column with one 16-byte load each (the sums still run over m in order);
// rows are padded by 4 floats so the 4 rows (and 8 columns) a warp reads
// fall in different banks.
constexpr int kScanCols = 16;
constexpr int kScanThreads = 256;
constexpr int kScanRowStep = kScanThreads / kScanCols;  // a thread's rows: c0 + kScanRowStep r

template <int D>
struct ScanSmem {
  static constexpr int LD = D + 4;
  float M[2][D * LD];
  float S[kScanCols * LD];  // S_in^T: [column][m]
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D>
__global__ void __launch_bounds__(kScanThreads)
segment_scan_kernel(PrefillArgs a) {
  extern __shared__ __align__(16) unsigned char scan_smem[];
  ScanSmem<D>& sm = *reinterpret_cast<ScanSmem<D>*>(scan_smem);
  constexpr int LD = ScanSmem<D>::LD;
  constexpr int RPT = D * kScanCols / kScanThreads;  // output rows per thread (4 or 2)
  const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * kScanCols;
  const int32_t n_segs = *a.plan.n_segs;
  __shared__ int32_t s_first, s_count;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_first = -1;
    s_count = 0;
    // binary search over segments for seq == n, index == 0 (segments are ordered by sequence)
    int lo = 0, hi = n_segs;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (!kda_guard(mid, 1, a.plan.capacity, a.err)) break;
      if (a.plan.segs[mid].seq < n) lo = mid + 1; else hi = mid;
    }
    if (lo < n_segs && kda_guard(lo, 1, a.plan.capacity, a.err) && a.plan.segs[lo].seq == n) {
      s_first = lo;
      s_count = a.plan.segs[lo].count;
    }
  }
  __syncthreads();
  // first_replayed: segment 0 was replayed in the first pass, which wrote
  // S_in(1); the chain starts there, so sequences of 2 segments need nothing
  // here.  Otherwise the chain starts from S0 with segment 0's record.
  const int j0 = a.plan.first_replayed ? 1 : 0;  // first segment chained here
  if (s_first < 0 || s_count <= 1 + j0) return;
  // records and entry states are D (128) wide; the caller's S0 is a.dv wide
  // (64 runs zero-padded to 128)
  const int W = 2 * D;  // width of the B | M record
  const int DIO = a.dv;
  // element offset of segment seg's record in incr_trans (n_it floats), and
  // the entry states' extent
  auto rec_off = [&](int64_t seg) { return (seg * a.H + h) * static_cast<int64_t>(D) * W; };
  const int64_t n_it = static_cast<int64_t>(a.plan.capacity) * a.H * D * W;
  const int64_t n_es = static_cast<int64_t>(a.plan.capacity) * a.H * D * D;
  auto stage_M = [&](int buf, int64_t off) {  // M_j -> sm.M[buf], 16 bytes per copy
    for (int i = tid; i < D * (D / 4); i += kScanThreads) {
      const int c = i / (D / 4), m4 = i % (D / 4);
      const int64_t e = off + static_cast<int64_t>(c) * W + D + 4 * m4;
      if (kda_guard(e, 4, n_it, a.err)) cp_async16(&sm.M[buf][c * LD + 4 * m4], a.incr_trans + e);
    }
    cp_async_commit();
  };
  stage_M(0, rec_off(s_first + j0));
  for (int i = tid; i < D * kScanCols; i += kScanThreads) {  // S_in(j0), transposed
    const int c = i / kScanCols, j = i % kScanCols;
    float& dst = sm.S[j * LD + c];
    if (j0) {
      const int64_t e = ((static_cast<int64_t>(s_first) + 1) * a.H + h) * static_cast<int64_t>(D) * D +
                        static_cast<int64_t>(c) * D + col0 + j;
      dst = kda_guard(e, 1, n_es, a.err) ? a.entry_state[e] : 0.f;
    } else {
      const int64_t e = ((static_cast<int64_t>(n) * a.H + h) * DIO + c) * DIO + col0 + j;
      dst = (a.S0 && c < DIO && col0 + j < DIO &&
             kda_guard(e, 1, static_cast<int64_t>(a.N) * a.H * DIO * DIO, a.err))
                ? a.S0[e]
                : 0.f;
    }
  }
  const int j = tid % kScanCols, c0 = tid / kScanCols;  // rows c0 + kScanRowStep r
  // B_j of this thread's outputs, loaded one segment ahead so its latency
  // overlaps the previous step
  float b_next[RPT];
  auto load_B = [&](int64_t seg) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int64_t e = rec_off(seg) + static_cast<int64_t>(c0 + kScanRowStep * r) * W + col0 + j;
      b_next[r] = kda_guard(e, 1, n_it, a.err) ? a.incr_trans[e] : 0.f;
    }
  };
  load_B(s_first + j0);
  for (int sgi = j0; sgi + 1 < s_count; ++sgi) {
    const int64_t seg = s_first + sgi;
    float acc[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) acc[r] = b_next[r];  // B_j
    if (sgi + 2 < s_count) load_B(seg + 1);
    if (sgi + 2 < s_count) {  // stage the next transition while this one is used
      stage_M((sgi - j0 + 1) & 1, rec_off(seg + 1));
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* Mb = sm.M[(sgi - j0) & 1];
    const float* Sj = sm.S + j * LD;
#pragma unroll 2
    for (int m = 0; m < D; m += 4) {
      const float4 s4 = *reinterpret_cast<const float4*>(Sj + m);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float4 m4 = *reinterpret_cast<const float4*>(Mb + (c0 + kScanRowStep * r) * LD + m);
        acc[r] = fmaf(m4.x, s4.x, acc[r]);
        acc[r] = fmaf(m4.y, s4.y, acc[r]);
        acc[r] = fmaf(m4.z, s4.z, acc[r]);
        acc[r] = fmaf(m4.w, s4.w, acc[r]);
      }
    }
    __syncthreads();  // every thread has read S_in(j) and this M buffer
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int c = c0 + kScanRowStep * r;
      sm.S[j * LD + c] = acc[r];
      const int64_t e = ((seg + 1) * a.H + h) * static_cast<int64_t>(D) * D +
                        static_cast<int64_t>(c) * D + col0 + j;
      if (kda_guard(e, 1, n_es, a.err)) a.entry_state[e] = acc[r];
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* cu_seqlens, int64_t T, int32_t N, int64_t L, Plan plan,
                        int* err, cudaStream_t s) {
  prof_begin(s, "kda_plan");
  plan_kernel<<<1, kPlanThreads, 0, s>>>(cu_seqlens, T, N, L, plan, err);
  prof_end(s, "kda_plan");
  return cudaGetLastError();
}

cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s) {
  // the chunk kernels keep 128-wide states for both head sizes
  dim3 grid(a.N, a.H, kStateD / kScanCols);
  prof_begin(s, "kda_segment_scan");
  cudaError_t e = cudaFuncSetAttribute(segment_scan_kernel<kStateD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(ScanSmem<kStateD>)));
  if (e == cudaSuccess)
    segment_scan_kernel<kStateD><<<grid, kScanThreads, sizeof(ScanSmem<kStateD>), s>>>(a);
  prof_end(s, "kda_segment_scan");
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kda
