"""ctypes binding of ``libkda.so`` (the C ABI in ``include/kda.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch supplies device memory and the current stream.  There is no
fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_PKG, "csrc")
_INCLUDE = os.path.join(os.path.dirname(_PKG), "include")
_BUILD = os.path.join(_PKG, "_build")
_LIB = os.path.join(_BUILD, "libkda.so")
# the bounds-checked build (-DKDA_BOUNDS_CHECK), objects and library apart
_BUILD_CHECKED = os.path.join(_BUILD, "checked")
_LIB_CHECKED = os.path.join(_BUILD_CHECKED, "libkda.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_libs = {}          # False: the normal library, True: the bounds-checked one
_checked = False    # which one load() returns

STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED",
          3: "KDA_ERR_CUDA", 4: "KDA_ERR_OUT_OF_MEMORY", 5: "KDA_ERR_DEVICE_INPUT"}


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_CHECKED if _checked else _LIB


def use_checked(checked: bool) -> None:
    """Route every call of this module to the bounds-checked library (True)
    or to the normal one (False, the default).  Both may be loaded at once;
    each keeps its own device state."""
    global _checked
    _checked = bool(checked)


def _sources():
    return sorted(os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(_INCLUDE, "kda.h")]


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile every ``csrc/*.cu`` for sm_103a and link ``_build/libkda.so``
    (with ``checked``: ``_build/checked/libkda.so``, every kernel compiled with
    -DKDA_BOUNDS_CHECK).

    Translation units compile in parallel; nvcc cross-compiles, so no GPU is
    needed.  Rebuilds only when a source or header is newer than the library.
    """
    bdir, lib_path = (_BUILD_CHECKED, _LIB_CHECKED) if checked else (_BUILD, _LIB)
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    newest = max(os.path.getmtime(p) for p in srcs + _headers())
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest:
        return lib_path
    common = ["nvcc", *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", _INCLUDE, "-I", _CSRC, "--expt-relaxed-constexpr"]
    if checked:
        common.append("-DKDA_BOUNDS_CHECK")
    objs, procs = [], []
    for src in srcs:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = common + ["-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out.decode(errors="replace"))
        if p.returncode:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call(["nvcc", *ARCH_FLAGS, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib_path)
    return lib_path


class KdaTensor(ctypes.Structure):
    """``kda_tensor`` of include/kda.h."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


KDA_DTYPE = {torch.bfloat16: 0, torch.float32: 1, torch.int32: 2}


def describe(t):
    """A kda_tensor for a torch tensor (None for None): pointer, dtype,
    shape and strides exactly as torch holds them, unchecked."""
    if t is None:
        return None
    d = KdaTensor()
    d.data = t.data_ptr()
    d.dtype = KDA_DTYPE.get(t.dtype, 99)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


def load():
    """Load (building first if needed) the library; returns the ctypes handle."""
    with _lock:
        if _checked not in _libs:
            path = library_path()
            if not os.path.exists(path):
                path = build(checked=_checked)
            lib = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            lib.kda_chunk_fwd.restype = ctypes.c_int
            lib.kda_chunk_fwd.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, vp]
            lib.kda_chunk_fwd_split.restype = ctypes.c_int
            lib.kda_chunk_fwd_split.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, i64, vp]
            lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
            lib.kda_chunk_fwd_noalloc.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, vp]
            lib.kda_decode_step.restype = ctypes.c_int
            lib.kda_decode_step.argtypes = [vp] * 7 + [i32, i32, i32, i32, vp]
            lib.kda_chunk_fwd_fused.restype = ctypes.c_int
            lib.kda_chunk_fwd_fused.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, vp]
            lib.kda_decode_step_fused.restype = ctypes.c_int
            lib.kda_decode_step_fused.argtypes = [vp] * 7 + [i32, i32, i32, i32, vp]
            lib.kda_chunk_fwd_checkpoints.restype = ctypes.c_int
            lib.kda_chunk_fwd_checkpoints.argtypes = ([vp] * 9 + [i64, i32, i32, i32, i32, i64, vp, i64, vp])
            lib.kda_chunk_fwd_host.restype = ctypes.c_int
            lib.kda_chunk_fwd_host.argtypes = [vp] * 8 + [i64, i32, i32, i32, i32, i64, vp]
            lib.kda_decode_tokens_fused.restype = ctypes.c_int
            lib.kda_decode_tokens_fused.argtypes = [vp] * 8 + [i32, i32, i32, i32, i32, vp]
            lib.kda_decode_tokens.restype = ctypes.c_int
            lib.kda_decode_tokens.argtypes = [vp] * 8 + [i32, i32, i32, i32, i32, vp]
            lib.kda_get_device_error.restype = ctypes.c_int
            lib.kda_get_device_error.argtypes = [vp]
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [ctypes.c_int]
            lib.kda_last_error_message.restype = ctypes.c_char_p
            lib.kda_last_error_message.argtypes = []
            lib.kda_abi_version.restype = ctypes.c_int
            tp = ctypes.POINTER(KdaTensor)
            lib.kda_chunk_fwd_t.restype = ctypes.c_int
            lib.kda_chunk_fwd_t.argtypes = [tp] * 9 + [vp]
            lib.kda_decode_step_t.restype = ctypes.c_int
            lib.kda_decode_step_t.argtypes = [tp] * 7 + [vp]
            lib.kda_debug_chunk_dump.restype = ctypes.c_int
            lib.kda_debug_chunk_dump.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, i32, i32, i64,
                                                         vp, vp]
            lib.kda_workspace_pool_bytes.restype = ctypes.c_int64
            lib.kda_workspace_pool_bytes.argtypes = []
            lib.kda_auto_segment_tokens.restype = ctypes.c_int64
            lib.kda_auto_segment_tokens.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int32, ctypes.c_int32]
            lib.kda_selftest_bounded_wait.restype = ctypes.c_int
            lib.kda_selftest_bounded_wait.argtypes = [ctypes.c_uint32, vp]
            lib.kda_selftest_bounds_check.restype = ctypes.c_int
            lib.kda_selftest_bounds_check.argtypes = [vp]
            lib.kda_bounds_checked.restype = ctypes.c_int
            lib.kda_bounds_checked.argtypes = []
            lib.kda_profile_enable.restype = None
            lib.kda_profile_enable.argtypes = [ctypes.c_int]
            lib.kda_profile_read.restype = ctypes.c_int
            lib.kda_profile_read.argtypes = [ctypes.POINTER(_KernelTime), ctypes.c_int]
            _libs[_checked] = lib
    return _libs[_checked]


def _check(status: int):
    if status != 0:
        msg = load().kda_last_error_message().decode(errors="replace")
        raise KdaError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise KdaError(1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise KdaError(1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise KdaError(1, f"{name} must be contiguous")


def kda_chunk_fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, out=None,
                  S_final=None, *, n_seqs=None, segment_tokens=0, want_state=True,
                  stream=None, _fused=False):
    """Prefill.  Tensors in the packed layout of ``include/kda.h``.

    q, k: bf16 [T, H, dk] (or [B, T_b, H, dk], a uniform batch); v bf16;
    log_alpha f32; beta f32 [T, H]; S0 f32 [N, H, dk, dv] or None;
    cu_seqlens int32 [N+1] (CUDA) or None.  Returns (out, S_final).
    """
    if q.dim() == 4:  # uniform batch [B, T_b, H, d]
        B = q.shape[0]
        q, k, v = (x.reshape(-1, *x.shape[2:]) for x in (q, k, v))
        log_alpha = log_alpha.reshape(-1, *log_alpha.shape[2:])
        beta = beta.reshape(-1, beta.shape[-1])
        if n_seqs is None:
            n_seqs = B
    T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.shape[0] - 1
    elif n_seqs is None:
        n_seqs = 1
    la_dt, la_name = (torch.bfloat16, "gate") if _fused else (torch.float32, "log_alpha")
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, la_dt, la_name),
                        (beta, torch.float32, "beta"), (S0, torch.float32, "S0"),
                        (cu_seqlens, torch.int32, "cu_seqlens")):
        _require(t, dt, name)
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    if S_final is None and want_state:
        S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out")
    _require(S_final, torch.float32, "S_final")
    lib = load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
            _ptr(cu_seqlens), _ptr(out), _ptr(S_final), T, n_seqs, H, dk, dv]
    if _fused:
        if segment_tokens:
            raise ValueError("the fused entry point chooses its own segments")
        _check(lib.kda_chunk_fwd_fused(*args, _stream(stream)))
    elif segment_tokens:
        _check(lib.kda_chunk_fwd_split(*args, int(segment_tokens), _stream(stream)))
    else:
        _check(lib.kda_chunk_fwd(*args, _stream(stream)))
    return out, S_final


def kda_chunk_fwd_fused(q_raw, k_raw, v, gate, beta, S0=None, cu_seqlens=None, out=None,
                        S_final=None, *, n_seqs=None, want_state=True, stream=None):
    """Prefill with the input preparation on load: q_raw, k_raw bf16 unnormalised,
    gate bf16 logits [T, H, dk] in place of log_alpha (log alpha = -5 sigmoid(gate)).
    Otherwise as :func:`kda_chunk_fwd`."""
    return kda_chunk_fwd(q_raw, k_raw, v, gate, beta, S0, cu_seqlens, out, S_final,
                         n_seqs=n_seqs, want_state=want_state, stream=stream, _fused=True)


def kda_decode_step(q, k, v, log_alpha, beta, S_inout, out=None, *, stream=None):
    """One decode step; ``S_inout`` [N, H, dk, dv] f32 is updated in place.

    q, k: bf16 [N, H, dk]; v bf16 [N, H, dv]; log_alpha f32 [N, H, dk];
    beta f32 [N, H].  Returns out bf16 [N, H, dv].
    """
    N, H, dk = q.shape
    dv = v.shape[-1]
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, torch.float32, "log_alpha"),
                        (beta, torch.float32, "beta"), (S_inout, torch.float32, "S_inout")):
        _require(t, dt, name)
    if out is None:
        out = torch.empty((N, H, dv), dtype=torch.bfloat16, device=q.device)
    _require(out, torch.bfloat16, "out")
    _check(load().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                  _ptr(S_inout), _ptr(out), N, H, dk, dv, _stream(stream)))
    return out


def kda_decode_step_fused(q_raw, k_raw, v, gate, beta, S_inout, out=None, *, stream=None):
    """Decode step with the input preparation on load (see :func:`kda_chunk_fwd_fused`)."""
    N, H, dk = q_raw.shape
    dv = v.shape[-1]
    for t, dt, name in ((q_raw, torch.bfloat16, "q_raw"), (k_raw, torch.bfloat16, "k_raw"),
                        (v, torch.bfloat16, "v"), (gate, torch.bfloat16, "gate"),
                        (beta, torch.float32, "beta"), (S_inout, torch.float32, "S_inout")):
        _require(t, dt, name)
    if out is None:
        out = torch.empty((N, H, dv), dtype=torch.bfloat16, device=q_raw.device)
    _require(out, torch.bfloat16, "out")
    _check(load().kda_decode_step_fused(_ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(gate),
                                        _ptr(beta), _ptr(S_inout), _ptr(out), N, H, dk, dv,
                                        _stream(stream)))
    return out


def _dref(d):
    return None if d is None else ctypes.byref(d)


def kda_chunk_fwd_t(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, out=None, S_final=None,
                    *, stream=None):
    """The descriptor form of the prefill: tensors go to the library with their
    dtype, shape and strides, and the library checks them.  ``out`` and
    ``S_final`` must be given (None skips S_final)."""
    descs = [describe(t) for t in (q, k, v, log_alpha, beta, S0, cu_seqlens, out, S_final)]
    _check(load().kda_chunk_fwd_t(*[_dref(d) for d in descs], _stream(stream)))
    return out, S_final


def kda_decode_step_t(q, k, v, log_alpha, beta, S_inout, out, *, stream=None):
    """The descriptor form of the decode step (see :func:`kda_chunk_fwd_t`)."""
    descs = [describe(t) for t in (q, k, v, log_alpha, beta, S_inout, out)]
    _check(load().kda_decode_step_t(*[_dref(d) for d in descs], _stream(stream)))
    return out


DUMP_LAYOUT = {"g": (0, (64, 128)), "A_kk": (8192, (64, 64)), "A_qk": (12288, (64, 64)),
               "T": (16384, (64, 64)), "U": (20480, (64, 128)), "S": (28672, (128, 128))}
DUMP_FLOATS = 45056


def kda_debug_chunk_dump(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, n_seqs=None,
                         seq, head, chunk, stream=None):
    """kda_chunk_fwd (never split) plus the intermediates of one chunk.

    Returns (out, S_final, {name: tensor}) with the names of DUMP_LAYOUT."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.shape[0] - 1
    elif n_seqs is None:
        n_seqs = 1
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, torch.float32, "log_alpha"),
                        (beta, torch.float32, "beta"), (S0, torch.float32, "S0"),
                        (cu_seqlens, torch.int32, "cu_seqlens")):
        _require(t, dt, name)
    out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    dump = torch.zeros(DUMP_FLOATS, dtype=torch.float32, device=q.device)
    _check(load().kda_debug_chunk_dump(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                       _ptr(S0), _ptr(cu_seqlens), _ptr(out), _ptr(S_final), T,
                                       n_seqs, H, dk, dv, int(seq), int(head), int(chunk),
                                       _ptr(dump), _stream(stream)))
    parts = {name: dump[off:off + int(np.prod(shape))].view(*shape)
             for name, (off, shape) in DUMP_LAYOUT.items()}
    return out, S_final, parts


def kda_auto_segment_tokens(total_tokens, n_seqs, n_heads, sm_count, uniform) -> int:
    """The segment length the automatic split picks (-1: no split); host only.
    ``uniform``: the batch has cu_seqlens None (sequences of equal length)."""
    return int(load().kda_auto_segment_tokens(total_tokens, n_seqs, n_heads, sm_count,
                                              1 if uniform else 0))


def kda_workspace_pool_bytes() -> int:
    """Bytes reserved by the library's workspace pool on the current device,
    or -1 when the library has created no pool there."""
    return int(load().kda_workspace_pool_bytes())


def kda_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return load().kda_get_device_error(_stream(stream))


def kda_bounds_checked() -> bool:
    """Whether the loaded library is the bounds-checked build."""
    return bool(load().kda_bounds_checked())


def kda_selftest_bounds_check(*, stream=None):
    """One out-of-range guard, no memory access (see include/kda.h)."""
    _check(load().kda_selftest_bounds_check(_stream(stream)))


def kda_selftest_bounded_wait(polls: int = 1000, *, stream=None):
    """One bounded wait on an mbarrier nothing arrives on (see include/kda.h);
    the next kda_get_device_error() reports the timeout."""
    _check(load().kda_selftest_bounded_wait(int(polls), _stream(stream)))


def profile_enable(on: bool = True):
    load().kda_profile_enable(1 if on else 0)


def profile_read():
    """{kernel name: (launches, total ms)} since the last read."""
    buf = (_KernelTime * 32)()
    n = load().kda_profile_read(buf, 32)
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(n)}


def kda_decode_tokens(q, k, v, log_alpha, beta, S_inout, commit=None, out=None, *, stream=None):
    """K tokens per sequence from the state ``S_inout`` [N, H, dk, dv] f32.

    q, k: bf16 [N, K, H, dk]; v bf16 [N, K, H, dv]; log_alpha f32 [N, K, H, dk];
    beta f32 [N, K, H]; commit: int32 [N] (CUDA) or None (commit all K).
    Returns out bf16 [N, K, H, dv]; ``S_inout`` holds the state after the
    committed tokens of each sequence.
    """
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, torch.float32, "log_alpha"),
                        (beta, torch.float32, "beta"), (S_inout, torch.float32, "S_inout"),
                        (commit, torch.int32, "commit")):
        _require(t, dt, name)
    if out is None:
        out = torch.empty((N, K, H, dv), dtype=torch.bfloat16, device=q.device)
    _require(out, torch.bfloat16, "out")
    _check(load().kda_decode_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                    _ptr(S_inout), _ptr(out), _ptr(commit), N, K, H, dk, dv,
                                    _stream(stream)))
    return out


def kda_chunk_fwd_checkpoints(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, interval,
                              max_checkpoints, n_seqs=None, stream=None):
    """Prefill that also returns the state after every ``interval`` tokens of each
    sequence (see include/kda.h).  Returns (out, S_final, checkpoints), checkpoints
    f32 [max_checkpoints, H, dk, dv] packed sequence by sequence."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.shape[0] - 1
    elif n_seqs is None:
        n_seqs = 1
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, torch.float32, "log_alpha"),
                        (beta, torch.float32, "beta"), (S0, torch.float32, "S0"),
                        (cu_seqlens, torch.int32, "cu_seqlens")):
        _require(t, dt, name)
    out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    ck = torch.empty((max(int(max_checkpoints), 1), H, dk, dv), dtype=torch.float32,
                     device=q.device)[:int(max_checkpoints)]
    _check(load().kda_chunk_fwd_checkpoints(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
        _ptr(out), _ptr(S_final), T, n_seqs, H, dk, dv, int(interval),
        _ptr(ck) if int(max_checkpoints) > 0 else None, int(max_checkpoints), _stream(stream)))
    return out, S_final, ck


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, S0, out, S_final, *, n_seqs, slice_tokens=0,
                       stream=None):
    """Prefill of a uniform batch held in HOST tensors (pin them for overlap).

    q, k, v, log_alpha, beta, out, S0 / S_final as in :func:`kda_chunk_fwd`, but CPU
    tensors; out and S_final are written once ``stream`` is synchronised."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    for t, dt, name in ((q, torch.bfloat16, "q"), (k, torch.bfloat16, "k"),
                        (v, torch.bfloat16, "v"), (log_alpha, torch.float32, "log_alpha"),
                        (beta, torch.float32, "beta"), (S0, torch.float32, "S0"),
                        (out, torch.bfloat16, "out"), (S_final, torch.float32, "S_final")):
        if t is None:
            continue
        if t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise KdaError(1, f"{name} must be a contiguous CPU {dt} tensor")
    _check(load().kda_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                     _ptr(S0), _ptr(out), _ptr(S_final), T, n_seqs, H, dk, dv,
                                     int(slice_tokens), _stream(stream)))
    return out, S_final


def kda_decode_tokens_fused(q_raw, k_raw, v, gate, beta, S_inout, commit=None, out=None, *,
                            stream=None):
    """:func:`kda_decode_tokens` with raw q, k and bf16 gate logits [N, K, H, dk]."""
    N, K, H, dk = q_raw.shape
    dv = v.shape[-1]
    for t, dt, name in ((q_raw, torch.bfloat16, "q_raw"), (k_raw, torch.bfloat16, "k_raw"),
                        (v, torch.bfloat16, "v"), (gate, torch.bfloat16, "gate"),
                        (beta, torch.float32, "beta"), (S_inout, torch.float32, "S_inout"),
                        (commit, torch.int32, "commit")):
        _require(t, dt, name)
    if out is None:
        out = torch.empty((N, K, H, dv), dtype=torch.bfloat16, device=q_raw.device)
    _require(out, torch.bfloat16, "out")
    _check(load().kda_decode_tokens_fused(_ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(gate),
                                          _ptr(beta), _ptr(S_inout), _ptr(out), _ptr(commit),
                                          N, K, H, dk, dv, _stream(stream)))
    return out
