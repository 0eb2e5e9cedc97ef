"""The C ABI on the host: the library builds for sm_103a, loads, exports every
entry point include/kda.h declares, and rejects bad arguments synchronously
before touching the GPU (these calls never reach a CUDA API, so they run
without a GPU)."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_48_gb300 import binding as kb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    kb.build()
    return kb.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("kda_chunk_fwd", "kda_decode_step", "kda_get_device_error",
                 "kda_status_string", "kda_last_error_message", "kda_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported by {kb.library_path()}"


def test_abi_version_and_status_strings(lib):
    assert lib.kda_abi_version() == 1
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(5) == b"KDA_ERR_DEVICE_INPUT"


# fake, 16-byte aligned, non-overlapping device addresses: validation rejects
# the call before any pointer is used
BASE = 1 << 40
STEP = 1 << 32


def P(i, off=0):
    return ctypes.c_void_p(BASE + i * STEP + off)


def prefill(lib, T=128, N=2, H=2, dk=64, dv=64, ptrs=None, seg=None, **over):
    p = {n: P(i) for i, n in enumerate(
        ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out", "S_final"])}
    p["cu_seqlens"] = None
    p.update(over)
    args = [p[n] for n in ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out",
                           "S_final"]] + [T, N, H, dk, dv]
    if seg is not None:
        return lib.kda_chunk_fwd_split(*args, seg, None)
    return lib.kda_chunk_fwd(*args, None)


def test_prefill_rejects_unsupported_head_sizes(lib):
    assert prefill(lib, dk=96, dv=96) == UNSUPPORTED
    assert prefill(lib, dk=128, dv=64) == UNSUPPORTED
    assert b"dk" in lib.kda_last_error_message()
    assert prefill(lib, dk=0, dv=0) == INVALID


@pytest.mark.parametrize("name", ["q", "k", "v", "log_alpha", "beta", "out"])
def test_prefill_rejects_null_required_pointer(lib, name):
    assert prefill(lib, **{name: None}) == INVALID
    assert name.encode() in lib.kda_last_error_message()


@pytest.mark.parametrize("name", ["q", "k", "v", "log_alpha", "beta", "S0", "out", "S_final"])
def test_prefill_rejects_misaligned_pointer(lib, name):
    idx = ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out", "S_final"].index(name)
    assert prefill(lib, **{name: P(idx, 8)}) == INVALID
    assert b"aligned" in lib.kda_last_error_message()


def test_prefill_rejects_bad_sizes(lib):
    assert prefill(lib, T=-1) == INVALID
    assert prefill(lib, N=0, T=10) == INVALID
    assert prefill(lib, H=0) == INVALID
    assert prefill(lib, T=129, N=2) == INVALID        # uniform batch must divide
    assert prefill(lib, seg=100) == INVALID            # segment not a multiple of 64


def test_prefill_rejects_more_heads_than_the_grid_allows(lib):
    # heads are the prefill kernels' second grid dimension: at most 65535
    assert prefill(lib, H=65536) == UNSUPPORTED
    assert b"n_heads" in lib.kda_last_error_message()
    a = [P(i) for i in range(9)]
    a[6] = None  # uniform batch
    assert lib.kda_chunk_fwd_noalloc(*a, 128, 2, 65536, 64, 64, None) == UNSUPPORTED
    assert lib.kda_chunk_fwd_host(*[P(i) for i in range(8)], 96, 3, 65536, 64, 64, 0,
                                  None) == UNSUPPORTED


def test_prefill_rejects_overlaps(lib):
    assert prefill(lib, out=P(0, 64)) == INVALID          # out inside q
    assert b"out overlaps" in lib.kda_last_error_message()
    assert prefill(lib, S_final=P(5, 16)) == INVALID      # partial overlap with S0
    assert prefill(lib, S_final=P(2)) == INVALID          # S_final over v
    assert prefill(lib, S_final=P(7, 16)) == INVALID      # S_final inside out


def test_prefill_empty_batch_is_a_noop(lib):
    assert prefill(lib, T=0, N=0) == OK


def decode(lib, N=4, H=2, dk=64, dv=64, **over):
    p = {n: P(i) for i, n in enumerate(["q", "k", "v", "log_alpha", "beta", "S", "out"])}
    p.update(over)
    return lib.kda_decode_step(p["q"], p["k"], p["v"], p["log_alpha"], p["beta"], p["S"],
                               p["out"], N, H, dk, dv, None)


def test_decode_rejects_bad_arguments(lib):
    assert decode(lib, dk=32, dv=32) == UNSUPPORTED
    assert decode(lib, S=None) == INVALID
    assert decode(lib, out=P(0, 4)) == INVALID            # misaligned
    assert decode(lib, out=P(5, 256)) == INVALID          # out inside the state
    assert decode(lib, S=P(0, 16)) == INVALID             # state overlaps q
    assert decode(lib, N=-1) == INVALID
    assert decode(lib, N=0) == OK


def test_build_targets_sm103a():
    assert "arch=compute_103a,code=sm_103a" in kb.ARCH_FLAGS


def fused_prefill(lib, T=128, N=2, H=2, dk=64, dv=64, **over):
    names = ["q", "k", "v", "gate", "beta", "S0", "cu_seqlens", "out", "S_final"]
    p = {n: P(i) for i, n in enumerate(names)}
    p["cu_seqlens"] = None
    p.update(over)
    return lib.kda_chunk_fwd_fused(*[p[n] for n in names], T, N, H, dk, dv, None)


def test_fused_entry_points_validate_like_the_plain_ones(lib):
    assert fused_prefill(lib, gate=None) == INVALID
    assert b"gate is NULL" in lib.kda_last_error_message()
    assert fused_prefill(lib, dk=96, dv=96) == UNSUPPORTED
    assert fused_prefill(lib, gate=P(3, 8)) == INVALID    # misaligned
    assert b"gate" in lib.kda_last_error_message()
    # the gate is bf16: T*H*dk*2 = 32 KiB, so `out` 40 KiB past its start is clear of it
    # but 24 KiB past it lands inside
    assert fused_prefill(lib, T=128, H=2, dk=64, out=P(3, 24 * 1024)) == INVALID
    assert b"out overlaps gate" in lib.kda_last_error_message()
    assert fused_prefill(lib, T=0, N=0) == OK
    args = [P(i) for i in range(7)]
    assert lib.kda_decode_step_fused(*args[:5], None, args[6], 4, 2, 64, 64, None) == INVALID
    assert lib.kda_decode_step_fused(*args, 4, 2, 32, 32, None) == UNSUPPORTED
    assert lib.kda_decode_step_fused(*args, 0, 2, 64, 64, None) == OK


def test_decode_tokens_validates_arguments(lib):
    a = [P(i) for i in range(8)]
    assert lib.kda_decode_tokens(*a, 4, 0, 2, 64, 64, None) == INVALID        # no tokens
    assert lib.kda_decode_tokens(*a[:7], P(7, 4), 4, 3, 2, 64, 64, None) == INVALID  # commit misaligned
    assert b"commit" in lib.kda_last_error_message()
    assert lib.kda_decode_tokens(*a[:6], P(7), P(7), 4, 3, 2, 64, 64, None) == INVALID  # out over commit
    assert lib.kda_decode_tokens(*a, 4, 3, 2, 96, 96, None) == UNSUPPORTED
    assert lib.kda_decode_tokens(*a, 0, 3, 2, 64, 64, None) == OK


def test_checkpoints_validate_arguments(lib):
    names = ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out", "S_final"]
    p = [P(i) for i in range(9)]
    p[6] = None

    def call(interval=128, ck=P(9), mx=4, T=256, N=2):
        return lib.kda_chunk_fwd_checkpoints(*p, T, N, 2, 64, 64, interval, ck, mx, None)

    assert call(interval=0) == INVALID
    assert call(interval=100) == INVALID                 # not a multiple of 64
    assert b"interval" in lib.kda_last_error_message()
    assert call(ck=None) == INVALID
    assert call(ck=P(9, 8)) == INVALID                   # misaligned
    assert call(ck=P(7, 64)) == INVALID                  # inside out
    assert b"checkpoints overlap" in lib.kda_last_error_message()
    assert call(T=0, N=0) == OK


def test_host_api_validates_arguments(lib):
    a = [P(i) for i in range(8)]
    assert lib.kda_chunk_fwd_host(*a, 100, 3, 2, 64, 64, 0, None) == INVALID   # not a multiple
    assert lib.kda_chunk_fwd_host(*a, 96, 3, 2, 64, 64, 100, None) == INVALID  # slice not x64
    assert lib.kda_chunk_fwd_host(*a, 96, 3, 2, 96, 96, 0, None) == UNSUPPORTED
    assert lib.kda_chunk_fwd_host(None, *a[1:], 96, 3, 2, 64, 64, 0, None) == INVALID
    assert lib.kda_chunk_fwd_host(*a, 0, 0, 2, 64, 64, 0, None) == OK


def test_selftest_rejects_bad_poll_counts(lib):
    # host-side checks only: nothing is launched
    assert lib.kda_selftest_bounded_wait(0, None) == 1  # KDA_ERR_INVALID_ARGUMENT
    assert lib.kda_selftest_bounded_wait((1 << 20) + 1, None) == 1


NAMES9 = ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out", "S_final"]

# (description, overrides of prefill()'s arguments): each call is invalid or
# unsupported for a reason found on the host
BAD_PREFILL_CALLS = [
    ("q misaligned", dict(q=P(0, 8))),
    ("beta misaligned", dict(beta=P(4, 4))),
    ("S_final misaligned", dict(S_final=P(8, 8))),
    ("cu_seqlens misaligned", dict(cu_seqlens=P(6, 4))),
    ("q missing", dict(q=None)),
    ("out missing", dict(out=None)),
    ("out inside q", dict(out=P(0, 64))),
    ("S_final over v", dict(S_final=P(2))),
    ("S_final partly over S0", dict(S_final=P(5, 16))),
    ("out over S_final", dict(out=P(8, 16))),
    ("dk != dv", dict(dk=128, dv=64)),
    ("dk = 96", dict(dk=96, dv=96)),
    ("dk = 0", dict(dk=0, dv=0)),
    ("uniform batch that does not divide", dict(T=129, N=2)),
    ("negative tokens", dict(T=-1)),
    ("tokens without sequences", dict(T=10, N=0)),
    ("no heads", dict(H=0)),
    ("too many heads", dict(H=65536)),
]


@pytest.mark.parametrize("what,over", BAD_PREFILL_CALLS, ids=[c[0] for c in BAD_PREFILL_CALLS])
def test_noalloc_rejects_what_kda_chunk_fwd_rejects(lib, what, over):
    """The no-allocation entry point applies kda_chunk_fwd's host checks: the
    same invalid call gets the same status (and a message) from both."""
    dims = {k: over.pop(k) for k in ("T", "N", "H", "dk", "dv") if k in over}
    full = dict(T=128, N=2, H=2, dk=64, dv=64)
    full.update(dims)
    p = {n: P(i) for i, n in enumerate(NAMES9)}
    p["cu_seqlens"] = None
    p.update(over)
    args = [p[n] for n in NAMES9] + [full["T"], full["N"], full["H"], full["dk"], full["dv"]]
    st_ref = lib.kda_chunk_fwd(*args, None)
    msg_ref = lib.kda_last_error_message()
    st = lib.kda_chunk_fwd_noalloc(*args, None)
    msg = lib.kda_last_error_message()
    assert st_ref in (INVALID, UNSUPPORTED), what
    assert st == st_ref, (what, msg_ref, msg)
    assert msg == msg_ref


def test_no_file_names_a_line_of_the_source_pages():
    """Sources are cited by page title and section, never by a line of the
    extracted page file."""
    bad = []
    for dirpath, dirs, files in os.walk(ROOT):
        dirs[:] = [d for d in dirs if not d.startswith((".", "_")) and d not in
                   ("gpurun_out", "baseline", "__pycache__")]
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".md", ".txt", ".json")):
                continue
            path = os.path.join(dirpath, f)
            rel = os.path.relpath(path, ROOT)
            if dirpath == ROOT and not f.endswith(".py"):
                continue  # top-level notes and records, several written by others
            with open(path, errors="replace") as fh:
                if "PAPER" + ".md" in fh.read():
                    bad.append(rel)
    assert not bad, bad
