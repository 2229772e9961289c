"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/gdn.h declares, sizes its buffers, and rejects
bad arguments with the right status before touching the device.  No call here
reaches a kernel launch."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_19_gb300 import _build, gdn

    _build.build()
    return gdn


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("gdn_fwd", "gdn_bwd", "gdn_fwd_workspace_bytes", "gdn_saved_bytes",
              "gdn_bwd_workspace_bytes", "gdn_status_string", "gdn_last_error", "gdn_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    handle = lib.load_library()
    for n in _declared_functions():
        assert hasattr(handle, n)


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gdn.h"\nint main(void){gdn_problem p={1,2,3,16,16,16,GDN_F32};'
                   'return (int)p.B - 1;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-c", str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_version_and_status_strings(lib):
    assert lib.gdn_version() >= 100
    assert lib.gdn_status_string(0) == "ok"
    assert "workspace" in lib.gdn_status_string(3)


def test_sizes(lib):
    p = lib.make_problem(8, 4096, 6, 128, 128, 64, 1)
    NC = 64
    # bf16 K=V=128 chunk 64 runs on tensor cores: bf16 boundary states followed by
    # the forward's chunk results (G f32; W, U, Mqk, T bf16), each region 256-aligned
    rows = 8 * 6 * NC * 64
    expect = 8 * 6 * NC * 128 * 128 * 2 + rows * 4 + rows * 128 * 2 * 2 + rows * 64 * 2 * 2
    assert lib.gdn_saved_bytes(p) == expect
    # bf16 K=V=64 chunk 64 also runs on tensor cores, with the same 128-wide buffers
    assert lib.gdn_saved_bytes(lib.make_problem(8, 4096, 6, 64, 64, 64, 1)) == expect
    # and so do K, V of 16 or 32, in any combination
    assert lib.gdn_saved_bytes(lib.make_problem(8, 4096, 6, 32, 16, 64, 1)) == expect
    assert lib.gdn_saved_bytes(lib.make_problem(8, 4096, 6, 16, 128, 64, 1)) == expect
    # other shapes keep float32 boundary states
    assert lib.gdn_saved_bytes(lib.make_problem(8, 4096, 6, 64, 64, 32, 1)) == 8 * 6 * 128 * 64 * 64 * 4
    assert lib.gdn_saved_bytes(lib.make_problem(8, 4096, 6, 64, 64, 64, 0)) == 8 * 6 * NC * 64 * 64 * 4
    assert lib.gdn_fwd_workspace_bytes(p) > 0
    assert lib.gdn_bwd_workspace_bytes(p) > lib.gdn_fwd_workspace_bytes(p)
    # ragged T rounds up to whole chunks
    p2 = lib.make_problem(1, 65, 1, 16, 16, 64, 0)
    assert lib.gdn_saved_bytes(p2) == 2 * 16 * 16 * 4
    # invalid problems size to 0
    assert lib.gdn_fwd_workspace_bytes(lib.make_problem(1, 8, 1, 24, 16, 16, 0)) == 0
    assert lib.gdn_saved_bytes(lib.make_problem(1, 8, 1, 16, 16, 48, 0)) == 0


FAKE = 1 << 40  # a 16-byte aligned address that is never dereferenced


def _fwd(lib, p, **over):
    h = lib.load_library()
    args = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), alpha=FAKE + (3 << 30),
                beta=FAKE + (4 << 30), s0=None, o=FAKE + (5 << 30), sT=None, saved=None,
                ws=FAKE + (6 << 30), ws_bytes=1 << 40)
    args.update(over)
    vp = ctypes.c_void_p
    return h.gdn_fwd(ctypes.byref(p), vp(args["q"]), vp(args["k"]), vp(args["v"]),
                     vp(args["alpha"]), vp(args["beta"]), vp(args["s0"]), vp(args["o"]),
                     vp(args["sT"]), vp(args["saved"]), vp(args["ws"]), args["ws_bytes"],
                     vp(None))


def _bwd(lib, p, **over):
    h = lib.load_library()
    base = dict(q=0, k=1, v=2, alpha=3, beta=4, s0=None, saved=None, do=5, dsT=None, dq=6,
                dk=7, dv=8, da=9, db=10, ds0=None, ws=11)
    args = {n: (None if x is None else FAKE + (x << 30)) for n, x in base.items()}
    args["ws_bytes"] = 1 << 40
    args.update(over)
    vp = ctypes.c_void_p
    order = ("q", "k", "v", "alpha", "beta", "s0", "saved", "do", "dsT", "dq", "dk", "dv",
             "da", "db", "ds0", "ws")
    return h.gdn_bwd(ctypes.byref(p), *[vp(args[n]) for n in order], args["ws_bytes"], vp(None))


def test_invalid_arguments_rejected_before_launch(lib):
    ok = lib.make_problem(2, 100, 3, 64, 32, 32, 1)
    INVALID, UNSUP, WS = 1, 2, 3
    assert _fwd(lib, lib.make_problem(1, 8, 1, 24, 16, 16, 1)) == UNSUP
    assert "K=24" in lib.gdn_last_error()
    assert _fwd(lib, lib.make_problem(1, 8, 1, 16, 16, 8, 1)) == UNSUP
    assert _fwd(lib, lib.make_problem(1, 8, 1, 16, 16, 16, 7)) == UNSUP
    assert _fwd(lib, lib.make_problem(-1, 8, 1, 16, 16, 16, 1)) == INVALID
    assert _fwd(lib, ok, q=None) == INVALID
    assert "q is NULL" in lib.gdn_last_error()
    assert _fwd(lib, ok, beta=FAKE + (4 << 30) + 8) == INVALID
    assert "aligned" in lib.gdn_last_error()
    assert _fwd(lib, ok, ws_bytes=16) == WS
    assert _fwd(lib, ok, o=FAKE + 64) == INVALID  # o overlaps q
    assert "overlaps" in lib.gdn_last_error()
    assert _fwd(lib, ok, sT=FAKE + (5 << 30) + 4096) == INVALID  # final_state inside o
    # bwd
    assert _bwd(lib, ok, do=None) == INVALID
    assert _bwd(lib, ok, dq=None) == INVALID
    assert _bwd(lib, ok, ws_bytes=0) == WS
    assert _bwd(lib, ok, dk=FAKE + (6 << 30) + 256) == INVALID  # dk overlaps dq
    assert _bwd(lib, ok, dv=FAKE) == INVALID  # dv overlaps q
    assert _bwd(lib, lib.make_problem(1, 8, 1, 16, 256, 16, 1)) == UNSUP
    # bf16 at chunk 64 runs on the tensor-core kernels, whose TMA row coordinates are
    # 32-bit: B*H*(ceil(T/64)+1)*128 must stay below 2^31 (the same token count in
    # float32 runs on the CUDA-core kernels, which index with 64 bits)
    big = lib.make_problem(64, 1 << 18, 256, 16, 16, 64, 1)
    assert _fwd(lib, big) == UNSUP
    assert "32-bit" in lib.gdn_last_error()
    assert lib.gdn_fwd_workspace_bytes(big) == 0
    assert _fwd(lib, lib.make_problem(64, 1 << 18, 256, 16, 16, 64, 0), ws_bytes=16) == WS
    edge = lib.make_problem(1, 64 * ((1 << 24) - 2), 1, 16, 16, 64, 1)  # (NC + 1) * 128 = 2^31 - 128
    assert lib.gdn_fwd_workspace_bytes(edge) > 0


def test_binding_refuses_cpu_tensors(lib):
    import torch

    q = torch.zeros(1, 4, 1, 16)
    with pytest.raises(lib.GdnError):
        lib.gdn_fwd(q, q, q, torch.ones(1, 4, 1), torch.zeros(1, 4, 1), chunk=16)


def _decode(lib, p, **over):
    h = lib.load_library()
    base = dict(q=0, k=1, v=2, alpha=3, beta=4, state=5, o=6)
    args = {n: FAKE + (x << 30) for n, x in base.items()}
    args.update(over)
    vp = ctypes.c_void_p
    order = ("q", "k", "v", "alpha", "beta", "state", "o")
    return h.gdn_decode(ctypes.byref(p), *[vp(args[n]) for n in order], vp(None))


def test_decode_arguments_rejected_before_launch(lib):
    INVALID, UNSUP = 1, 2
    ok = lib.make_problem(2, 1, 3, 64, 32, 64, 1)
    assert _decode(lib, ok, state=None) == INVALID
    assert "state is NULL" in lib.gdn_last_error()
    assert _decode(lib, ok, o=FAKE + (5 << 30)) == INVALID  # o is the state
    assert _decode(lib, ok, q=FAKE + 8) == INVALID          # misaligned
    assert _decode(lib, lib.make_problem(1, 1, 1, 24, 16, 64, 1)) == UNSUP
    # the chunk field is not used by the decode step: with T = 0 nothing launches
    assert _decode(lib, lib.make_problem(1, 0, 1, 16, 16, 7, 1)) == 0


def _varlen_fwd(lib, p, total, **over):
    h = lib.load_library()
    base = dict(cu=12, q=0, k=1, v=2, alpha=3, beta=4, s0=None, o=5, sT=None, saved=None, ws=6)
    args = {n: (None if x is None else FAKE + (x << 30)) for n, x in base.items()}
    args["ws_bytes"] = 1 << 40
    args.update(over)
    vp = ctypes.c_void_p
    order = ("cu", "q", "k", "v", "alpha", "beta", "s0", "o", "sT", "saved", "ws")
    return h.gdn_varlen_fwd(ctypes.byref(p), total, *[vp(args[n]) for n in order], args["ws_bytes"],
                            vp(None))


def _varlen_bwd(lib, p, total, **over):
    h = lib.load_library()
    base = dict(cu=13, q=0, k=1, v=2, alpha=3, beta=4, s0=None, saved=None, do=5, dsT=None, dq=6,
                dk=7, dv=8, da=9, db=10, ds0=None, ws=11)
    args = {n: (None if x is None else FAKE + (x << 30)) for n, x in base.items()}
    args["ws_bytes"] = 1 << 40
    args.update(over)
    vp = ctypes.c_void_p
    order = ("cu", "q", "k", "v", "alpha", "beta", "s0", "saved", "do", "dsT", "dq", "dk", "dv",
             "da", "db", "ds0", "ws")
    return h.gdn_varlen_bwd(ctypes.byref(p), total, *[vp(args[n]) for n in order], args["ws_bytes"],
                            vp(None))


def test_varlen_arguments_rejected_before_launch(lib):
    INVALID, UNSUP, WS = 1, 2, 3
    p = lib.make_problem(3, 100, 2, 64, 64, 64, 1)  # 3 sequences of at most 100 tokens
    assert _varlen_fwd(lib, p, 301) == INVALID  # more rows than 3 sequences can hold
    assert "total" in lib.gdn_last_error()
    assert _varlen_fwd(lib, p, -1) == INVALID
    assert _varlen_fwd(lib, p, 200, cu=None) == INVALID
    assert "cu_seqlens" in lib.gdn_last_error()
    assert _varlen_fwd(lib, p, 200, cu=FAKE + (12 << 30) + 2) == INVALID  # not 4-byte aligned
    assert _varlen_fwd(lib, p, 200, q=None) == INVALID
    assert _varlen_fwd(lib, p, 200, ws_bytes=1024) == WS
    need = lib.load_library().gdn_varlen_fwd_workspace_bytes(ctypes.byref(p), 200)
    assert need > 0
    assert _varlen_fwd(lib, p, 200, ws_bytes=need - 1) == WS
    assert _varlen_fwd(lib, p, 200, o=FAKE + 256) == INVALID          # o overlaps q
    assert _varlen_fwd(lib, p, 200, cu=FAKE + (5 << 30) + 64) == INVALID  # cu inside o
    assert _varlen_fwd(lib, p, 200, sT=FAKE + (5 << 30)) == INVALID   # final state is o
    assert _varlen_fwd(lib, lib.make_problem(3, 100, 2, 24, 64, 64, 1), 200) == UNSUP
    assert _varlen_bwd(lib, p, 200, do=None) == INVALID
    assert _varlen_bwd(lib, p, 200, dv=FAKE) == INVALID               # dv overlaps q
    assert _varlen_bwd(lib, p, 200, ds0=FAKE + (6 << 30)) == INVALID  # d_initial_state is dq
    assert _varlen_bwd(lib, p, 200, ws_bytes=0) == WS
    assert _varlen_bwd(lib, p, 301) == INVALID


def test_sequence_split_policy(lib):
    h = lib.load_library()
    INVALID = 1
    assert h.gdn_set_sequence_split(-1) == INVALID
    assert h.gdn_set_sequence_split(2000) == INVALID
    few = lib.make_problem(1, 2048, 2, 128, 128, 64, 1)   # 2 streams: the automatic policy splits
    many = lib.make_problem(8, 4096, 6, 128, 128, 64, 1)  # 48 streams: it does not
    try:
        assert h.gdn_set_sequence_split(1) == 0 and h.gdn_get_sequence_split() == 1
        off_f = h.gdn_fwd_workspace_bytes(ctypes.byref(few))
        off_b = h.gdn_bwd_workspace_bytes(ctypes.byref(few))
        off_many = h.gdn_fwd_workspace_bytes(ctypes.byref(many))
        assert h.gdn_set_sequence_split(0) == 0
        assert h.gdn_fwd_workspace_bytes(ctypes.byref(few)) > off_f  # piece states and transitions
        assert h.gdn_bwd_workspace_bytes(ctypes.byref(few)) > off_b
        assert h.gdn_fwd_workspace_bytes(ctypes.byref(many)) == off_many
        saved = h.gdn_saved_bytes(ctypes.byref(few))
        assert h.gdn_set_sequence_split(5) == 0
        assert h.gdn_saved_bytes(ctypes.byref(few)) == saved  # the split keeps nothing extra
        # B > 1 with T not a multiple of the chunk: the rows are not whole chunks apart, no split
        ragged = lib.make_problem(2, 100, 2, 128, 128, 64, 1)
        w5 = h.gdn_fwd_workspace_bytes(ctypes.byref(ragged))
        assert h.gdn_set_sequence_split(1) == 0
        assert h.gdn_fwd_workspace_bytes(ctypes.byref(ragged)) == w5
    finally:
        h.gdn_set_sequence_split(0)


def test_count_nonfinite_rejects_bad_arguments(lib):
    """Rejections return before any launch (and n = 0 launches nothing)."""
    h = lib.load_library()
    OK, INVALID, UNSUPPORTED = 0, 1, 2
    x, c = ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 20))
    assert h.gdn_count_nonfinite(x, -1, 0, c, None) == INVALID
    assert h.gdn_count_nonfinite(x, 10, 7, c, None) == UNSUPPORTED
    assert h.gdn_count_nonfinite(x, 10, 0, None, None) == INVALID
    assert h.gdn_count_nonfinite(x, 10, 0, ctypes.c_void_p(FAKE + 4), None) == INVALID  # count misaligned
    assert h.gdn_count_nonfinite(None, 10, 1, c, None) == INVALID
    assert h.gdn_count_nonfinite(ctypes.c_void_p(FAKE + 8), 10, 1, c, None) == INVALID  # x misaligned
    assert h.gdn_count_nonfinite(None, 0, 1, c, None) == OK


def _prologue(lib, p, bwd=False, **over):
    """gdn_prologue_fwd / _bwd on fake, disjoint, 16-byte aligned addresses (1 GB apart)."""
    h = lib.load_library()
    names = (("q_raw", "k_raw", "a", "b", "dq", "dk", "dalpha", "dbeta", "dq_raw", "dk_raw", "da", "db") if bwd
             else ("q_raw", "k_raw", "a", "b", "q", "k", "alpha", "beta"))
    args = {n: FAKE + (i << 30) for i, n in enumerate(names)}
    args.update(over)
    fn = h.gdn_prologue_bwd if bwd else h.gdn_prologue_fwd
    return fn(ctypes.byref(p), *[ctypes.c_void_p(args[n]) for n in names], ctypes.c_void_p(None))


@pytest.mark.parametrize("bwd", [False, True])
def test_prologue_arguments_rejected_before_launch(lib, bwd):
    INVALID, UNSUP = 1, 2
    ok = lib.make_problem(2, 5, 3, 64, 64, 64, 1)
    assert _prologue(lib, ok, bwd, q_raw=None) == INVALID
    assert "q_raw is NULL" in lib.gdn_last_error()
    assert _prologue(lib, ok, bwd, k_raw=FAKE + (1 << 30) + 8) == INVALID  # misaligned
    out = "dq_raw" if bwd else "q"
    assert _prologue(lib, ok, bwd, **{out: FAKE}) == INVALID  # an output on an input
    assert "overlaps" in lib.gdn_last_error()
    assert _prologue(lib, lib.make_problem(2, 5, 3, 24, 24, 64, 1), bwd) == UNSUP
    # no rows: every pointer may be NULL and nothing launches
    empty = lib.make_problem(2, 0, 3, 64, 64, 64, 1)
    names = 12 if bwd else 8
    h = lib.load_library()
    fn = h.gdn_prologue_bwd if bwd else h.gdn_prologue_fwd
    assert fn(ctypes.byref(empty), *([ctypes.c_void_p(None)] * names), ctypes.c_void_p(None)) == 0


def _raw(lib, p, bwd=False, **over):
    """gdn_fwd_raw / gdn_bwd_raw on fake, disjoint, 16-byte aligned addresses."""
    h = lib.load_library()
    if bwd:
        base = dict(q=0, k=1, v=2, a=3, b=4, s0=None, saved=None, do=5, dsT=None, dq=6, dk=7, dv=8, da=9,
                    db=10, ds0=None, ws=11)
        order = ("q", "k", "v", "a", "b", "s0", "saved", "do", "dsT", "dq", "dk", "dv", "da", "db", "ds0", "ws")
        fn = h.gdn_bwd_raw
    else:
        base = dict(q=0, k=1, v=2, a=3, b=4, s0=None, o=5, sT=None, saved=None, ws=6)
        order = ("q", "k", "v", "a", "b", "s0", "o", "sT", "saved", "ws")
        fn = h.gdn_fwd_raw
    args = {n: (None if x is None else FAKE + (x << 30)) for n, x in base.items()}
    args["ws_bytes"] = 1 << 40
    args.update(over)
    vp = ctypes.c_void_p
    return fn(ctypes.byref(p), *[vp(args[n]) for n in order], args["ws_bytes"], vp(None))


@pytest.mark.parametrize("bwd", [False, True])
def test_raw_arguments_rejected_before_launch(lib, bwd):
    INVALID, UNSUP, WS = 1, 2, 3
    for p in (lib.make_problem(2, 100, 3, 128, 128, 64, 1),   # tensor-core kernels, prologue folded in
              lib.make_problem(2, 100, 3, 64, 32, 32, 0)):    # prologue kernel, then the recurrence
        assert _raw(lib, p, bwd, q=None) == INVALID
        assert "q_raw is NULL" in lib.gdn_last_error()
        assert _raw(lib, p, bwd, b=FAKE + (4 << 30) + 8) == INVALID
        assert "aligned" in lib.gdn_last_error()
        assert _raw(lib, p, bwd, ws_bytes=16) == WS
        out = "dq" if bwd else "o"
        assert _raw(lib, p, bwd, **{out: FAKE + 64}) == INVALID  # an output on q_raw
        assert "overlaps" in lib.gdn_last_error()
    assert _raw(lib, lib.make_problem(1, 8, 1, 24, 16, 16, 1), bwd) == UNSUP


def test_raw_sizes(lib):
    tc = lib.make_problem(8, 4096, 6, 128, 128, 64, 1)
    BTH = 8 * 4096 * 6
    # the normalised q, k rows (bf16) and their reciprocal norms (fp32), then gdn_fwd's saved
    raw_part = 2 * BTH * 128 * 2 + 2 * BTH * 4
    assert lib.gdn_raw_saved_bytes(tc) == raw_part + lib.gdn_saved_bytes(tc)
    assert lib.gdn_raw_fwd_workspace_bytes(tc) == raw_part + lib.gdn_fwd_workspace_bytes(tc)
    # the backward also keeps one float per token for the k normalisation's chain rule
    assert lib.gdn_raw_bwd_workspace_bytes(tc) == raw_part + BTH * 4 + lib.gdn_bwd_workspace_bytes(tc)
    # other shapes keep gdn_fwd's saved; the workspace holds the prologue's outputs
    # (and, backward, the recurrence's input gradients) in the run dtype
    f = lib.make_problem(2, 100, 3, 64, 32, 32, 0)
    BTH = 2 * 100 * 3
    r = lambda x: (x + 255) // 256 * 256
    fwd_part = 2 * r(BTH * 64 * 4) + 2 * r(BTH * 4)
    assert lib.gdn_raw_saved_bytes(f) == lib.gdn_saved_bytes(f)
    assert lib.gdn_raw_fwd_workspace_bytes(f) == fwd_part + lib.gdn_fwd_workspace_bytes(f)
    assert lib.gdn_raw_bwd_workspace_bytes(f) == 2 * fwd_part + lib.gdn_bwd_workspace_bytes(f)
    assert lib.gdn_raw_fwd_workspace_bytes(lib.make_problem(1, 8, 1, 24, 16, 16, 0)) == 0


def _reset(lib, p, S_max, bwd=False, **over):
    """gdn_reset_fwd / gdn_reset_bwd on fake, disjoint, 16-byte aligned addresses."""
    h = lib.load_library()
    if bwd:
        base = dict(mask=12, q=0, k=1, v=2, a=3, b=4, s0=None, saved=None, do=5, dsT=None, dq=6, dk=7, dv=8, da=9,
                    db=10, ds0=None, ws=11)
        order = ("mask", "q", "k", "v", "a", "b", "s0", "saved", "do", "dsT", "dq", "dk", "dv", "da", "db", "ds0",
                 "ws")
        fn = h.gdn_reset_bwd
    else:
        base = dict(mask=12, q=0, k=1, v=2, a=3, b=4, s0=None, o=5, sT=None, saved=None, ws=6)
        order = ("mask", "q", "k", "v", "a", "b", "s0", "o", "sT", "saved", "ws")
        fn = h.gdn_reset_fwd
    args = {n: (None if x is None else FAKE + (x << 30)) for n, x in base.items()}
    args["ws_bytes"] = 1 << 40
    args.update(over)
    vp = ctypes.c_void_p
    return fn(ctypes.byref(p), S_max, *[vp(args[n]) for n in order], args["ws_bytes"], vp(None))


@pytest.mark.parametrize("bwd", [False, True])
def test_reset_arguments_rejected_before_launch(lib, bwd):
    INVALID, WS = 1, 3
    p = lib.make_problem(3, 100, 2, 128, 128, 64, 1)
    assert _reset(lib, p, 6, bwd, mask=None) == INVALID
    assert "reset is NULL" in lib.gdn_last_error()
    assert _reset(lib, p, 2, bwd) == INVALID  # fewer than one segment per row
    assert "max_segments" in lib.gdn_last_error()
    assert _reset(lib, p, 301, bwd) == INVALID  # more than B*T
    assert _reset(lib, p, 6, bwd, ws_bytes=64) == WS
    assert _reset(lib, p, 6, bwd, q=None) == INVALID  # the packed call's own checks
    h = lib.load_library()
    size = h.gdn_reset_bwd_workspace_bytes if bwd else h.gdn_reset_fwd_workspace_bytes
    assert size(ctypes.byref(p), 6) > 0
    assert size(ctypes.byref(p), 2) == 0
    assert h.gdn_reset_saved_bytes(ctypes.byref(p), 6) == h.gdn_varlen_saved_bytes(
        ctypes.byref(lib.make_problem(6, 100, 2, 128, 128, 64, 1)), 300)
