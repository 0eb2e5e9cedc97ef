// Descriptor form of the two layer calls (include/kda.h: kda_tensor,
// kda_chunk_fwd_t, kda_decode_step_t).  Each tensor travels with its dtype,
// shape and strides, so the library itself rejects a wrong dtype, an
// inconsistent shape or a non-dense layout before anything is launched.  The
// checked call then goes to the pointer entry point, which runs the kernels.
#include <cuda_runtime.h>

#include <cstdio>

#include "kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

const char* dtype_name(kda_dtype t) {
  switch (t) {
    case KDA_BF16: return "bf16";
    case KDA_F32: return "f32";
    case KDA_I32: return "i32";
  }
  return "unknown";
}

kda_status bad(const char* fmt, const char* name, long long a = 0, long long b = 0,
               long long c = 0) {
  char msg[256];
  snprintf(msg, sizeof msg, fmt, name, a, b, c);
  return report_error(KDA_ERR_INVALID_ARGUMENT, msg);
}

// dtype, rank, shape (entries < 0 in `want` are free) and dense row-major
// strides (in elements; a dimension of extent 1 may have any stride).
kda_status check_tensor(const kda_tensor* t, const char* name, kda_dtype dtype, int ndim,
                        const int64_t* want) {
  if (!t) return bad("%s: descriptor is NULL", name);
  if (t->dtype != dtype) {
    char msg[160];
    snprintf(msg, sizeof msg, "%s: dtype must be %s (got %s)", name, dtype_name(dtype),
             dtype_name(t->dtype));
    return report_error(KDA_ERR_INVALID_ARGUMENT, msg);
  }
  if (t->ndim != ndim) return bad("%s: must have %lld dimensions (got %lld)", name, ndim, t->ndim);
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return bad("%s: negative extent in dimension %lld", name, i);
    if (want[i] >= 0 && t->shape[i] != want[i])
      return bad("%s: dimension %lld is %lld, expected %lld", name, i, t->shape[i], want[i]);
  }
  int64_t expect = 1;
  for (int i = ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != expect)
      return bad("%s: not dense row-major (stride of dimension %lld is %lld, expected %lld)",
                 name, i, t->stride[i], expect);
    expect *= t->shape[i];
  }
  return KDA_OK;
}

kda_status check_optional(const kda_tensor* t, const char* name, kda_dtype dtype, int ndim,
                          const int64_t* want) {
  return t ? check_tensor(t, name, dtype, ndim, want) : KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_chunk_fwd_t(const kda_tensor* q, const kda_tensor* k,
                                      const kda_tensor* v, const kda_tensor* log_alpha,
                                      const kda_tensor* beta, const kda_tensor* S0,
                                      const kda_tensor* cu_seqlens, kda_tensor* out,
                                      kda_tensor* S_final, void* stream) {
  NvtxRange nvtx_range("kda_chunk_fwd_t");
  if (!q) return bad("%s: descriptor is NULL", "q");
  if (q->ndim != 3 && q->ndim != 4)
    return bad("%s: must be [T, H, dk] or [B, T_b, H, dk] (got %lld dimensions)", "q", q->ndim);
  const bool batched = q->ndim == 4;
  const int r = batched ? 1 : 0;  // index shift of [.., H, d] in a batched tensor
  const int64_t B = batched ? q->shape[0] : 0;
  const int64_t Tb = q->shape[r];
  const int64_t T = batched ? B * Tb : Tb;
  const int64_t H = q->shape[r + 1], dk = q->shape[r + 2];
  if (batched && cu_seqlens)
    return bad("%s: must be NULL for a [B, T_b, H, dk] batch", "cu_seqlens");
  const int64_t dv = v ? v->shape[q->ndim - 1] : -1;
  // number of sequences: B, the length of cu_seqlens minus one, else the
  // leading extent of S0 or S_final, else 1
  int64_t N = 1;
  if (batched) N = B;
  else if (cu_seqlens) N = cu_seqlens->shape[0] - 1;
  else if (S0) N = S0->shape[0];
  else if (S_final) N = S_final->shape[0];
  if (N < 0) return bad("%s: needs at least one entry", "cu_seqlens");
  if (cu_seqlens && cu_seqlens->ndim == 1)
    for (const kda_tensor* st : {S0, static_cast<const kda_tensor*>(S_final)})
      if (st && st->ndim == 4 && st->shape[0] != N)
        return bad("%s: %lld entries give %lld sequences, but the state has %lld", "cu_seqlens",
                   cu_seqlens->shape[0], N, st->shape[0]);
  const int nd = q->ndim;
  const int64_t sq[4] = {q->shape[0], q->shape[1], q->shape[2], nd == 4 ? q->shape[3] : 0};
  int64_t sv[4] = {sq[0], sq[1], sq[2], sq[3]};
  sv[nd - 1] = dv;
  const int64_t sb[4] = {sq[0], sq[1], nd == 4 ? sq[2] : 0, 0};
  const int64_t ss[4] = {N, H, dk, dv};
  const int64_t sc[1] = {N + 1};
  kda_status st;
  if ((st = check_tensor(q, "q", KDA_BF16, nd, sq)) != KDA_OK) return st;
  if ((st = check_tensor(k, "k", KDA_BF16, nd, sq)) != KDA_OK) return st;
  if ((st = check_tensor(v, "v", KDA_BF16, nd, sv)) != KDA_OK) return st;
  if ((st = check_tensor(log_alpha, "log_alpha", KDA_F32, nd, sq)) != KDA_OK) return st;
  if ((st = check_tensor(beta, "beta", KDA_F32, nd - 1, sb)) != KDA_OK) return st;
  if ((st = check_optional(S0, "S0", KDA_F32, 4, ss)) != KDA_OK) return st;
  if ((st = check_optional(cu_seqlens, "cu_seqlens", KDA_I32, 1, sc)) != KDA_OK) return st;
  if ((st = check_tensor(out, "out", KDA_BF16, nd, sv)) != KDA_OK) return st;
  if ((st = check_optional(S_final, "S_final", KDA_F32, 4, ss)) != KDA_OK) return st;
  if (N > 0x7fffffffLL || H > 0x7fffffffLL || dk > 0x7fffffffLL || dv > 0x7fffffffLL)
    return report_error(KDA_ERR_UNSUPPORTED, "an extent exceeds the int32 range");
  return kda_chunk_fwd(q->data, k->data, v->data, static_cast<const float*>(log_alpha->data),
                       static_cast<const float*>(beta->data),
                       S0 ? static_cast<const float*>(S0->data) : nullptr,
                       cu_seqlens ? static_cast<const int32_t*>(cu_seqlens->data) : nullptr,
                       out->data, S_final ? static_cast<float*>(S_final->data) : nullptr, T,
                       static_cast<int32_t>(N), static_cast<int32_t>(H),
                       static_cast<int32_t>(dk), static_cast<int32_t>(dv), stream);
}

extern "C" kda_status kda_decode_step_t(const kda_tensor* q, const kda_tensor* k,
                                        const kda_tensor* v, const kda_tensor* log_alpha,
                                        const kda_tensor* beta, kda_tensor* S_inout,
                                        kda_tensor* out, void* stream) {
  NvtxRange nvtx_range("kda_decode_step_t");
  if (!q) return bad("%s: descriptor is NULL", "q");
  if (q->ndim != 3) return bad("%s: must be [N, H, dk] (got %lld dimensions)", "q", q->ndim);
  const int64_t N = q->shape[0], H = q->shape[1], dk = q->shape[2];
  const int64_t dv = v ? v->shape[2] : -1;
  const int64_t sq[3] = {N, H, dk}, sv[3] = {N, H, dv}, sb[2] = {N, H};
  const int64_t ss[4] = {N, H, dk, dv};
  kda_status st;
  if ((st = check_tensor(q, "q", KDA_BF16, 3, sq)) != KDA_OK) return st;
  if ((st = check_tensor(k, "k", KDA_BF16, 3, sq)) != KDA_OK) return st;
  if ((st = check_tensor(v, "v", KDA_BF16, 3, sv)) != KDA_OK) return st;
  if ((st = check_tensor(log_alpha, "log_alpha", KDA_F32, 3, sq)) != KDA_OK) return st;
  if ((st = check_tensor(beta, "beta", KDA_F32, 2, sb)) != KDA_OK) return st;
  if ((st = check_tensor(S_inout, "S_inout", KDA_F32, 4, ss)) != KDA_OK) return st;
  if ((st = check_tensor(out, "out", KDA_BF16, 3, sv)) != KDA_OK) return st;
  if (N > 0x7fffffffLL || H > 0x7fffffffLL || dk > 0x7fffffffLL || dv > 0x7fffffffLL)
    return report_error(KDA_ERR_UNSUPPORTED, "an extent exceeds the int32 range");
  return kda_decode_step(q->data, k->data, v->data, static_cast<const float*>(log_alpha->data),
                         static_cast<const float*>(beta->data), static_cast<float*>(S_inout->data),
                         out->data, static_cast<int32_t>(N), static_cast<int32_t>(H),
                         static_cast<int32_t>(dk), static_cast<int32_t>(dv), stream);
}
