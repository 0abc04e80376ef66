"""The C-ABI library: it loads, exports exactly what include/kda.h declares, and rejects
bad arguments on the host before any launch (no GPU needed: every call below fails
validation, or needs no device work, so no CUDA call is made)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

OK, INVALID, UNSUPPORTED = 0, 1, 2
F32, BF16 = 0, 1


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names |= set(re.findall(r"^\s*(?:kda_status|size_t|int|const char\s*\*)\s*(kda_\w+)\s*\(",
                                text, flags=re.M))
    return names


@pytest.fixture(scope="session")
def lib():
    from chunked_kda_gb300 import _build

    path = _build.build()
    L = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.kda_chunk_fwd.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp, vp, i32,
                                i32, i32, i32, i32, i32, i32, vp, i32, vp, ctypes.c_size_t, vp]
    L.kda_recurrent_fwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                    i32, vp, i32, vp]
    L.kda_gate_fwd.argtypes = [vp, i32, vp, vp, i32, f32, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    L.kda_chunk_workspace_bytes.argtypes = [i32] * 8
    L.kda_chunk_workspace_bytes.restype = ctypes.c_size_t
    L.kda_chunk_workspace_bytes_ex.argtypes = [i32] * 9
    L.kda_chunk_workspace_bytes_ex.restype = ctypes.c_size_t
    L.kda_chunk_fwd_launches.argtypes = [i32] * 10
    L.kda_chunk_fwd_launches.restype = i32
    # full prototypes: a call with the wrong arity raises instead of passing stray values
    L.kda_chunk_fwd_ex.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp, vp, i32,
                                   i32, i32, i32, i32, i32, i32, vp, i32, vp, ctypes.c_size_t, i32,
                                   ctypes.c_uint, vp, vp]
    L.kda_test_hooks.argtypes = [i32, i32, i32, i32]
    L.kda_recurrent_fwd_ex.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp, vp,
                                       i32, i32, i32, i32, i32, i32, vp, i32, i32, ctypes.c_uint,
                                       vp]
    L.kda_chunk_fwd_noalloc.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp, vp,
                                        i32, i32, i32, i32, i32, i32, i32, vp, i32, vp]
    L.kda_status_string.restype = ctypes.c_char_p
    L.kda_last_error.restype = ctypes.c_char_p
    return L


def test_header_declares_the_entry_points():
    assert {"kda_gate_fwd", "kda_chunk_workspace_bytes", "kda_chunk_fwd", "kda_recurrent_fwd",
            "kda_status_string", "kda_last_error"} <= declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.skipif(shutil.which("nm") is None, reason="nm not available")
def test_no_undeclared_kda_exports():
    from chunked_kda_gb300 import _build

    out = subprocess.run(["nm", "-D", "--defined-only", _build.build()], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split() and
                ln.split()[-1].startswith("kda_")}
    assert exported == declared_functions()


def test_status_strings(lib):
    for code in range(4):
        assert lib.kda_status_string(code).startswith(b"KDA_")


def test_wait_timeouts_null_count(lib):
    """The diagnostics query rejects a null count on the host (no device access)."""
    lib.kda_fused_wait_timeouts.argtypes = [ctypes.c_void_p, ctypes.c_int]
    assert lib.kda_fused_wait_timeouts(None, 0) == 1  # KDA_ERR_INVALID_ARG


P = ctypes.c_void_p(4096)  # aligned stand-in: never dereferenced, validation fails first


def _chunk(lib, **kw):
    a = dict(q=P, k=P, v=P, dt=BF16, g=P, gdt=BF16, A_log=P, dt_bias=None, mode=1, lb=-5.0,
             beta=P, h0=None, hT=None, cu=None, n=0, B=1, T=64, H=2, K=128, V=128, C=64, o=P,
             odt=None, ws=None, ws_bytes=0)
    a.update(kw)
    if a["odt"] is None:
        a["odt"] = a["dt"]
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["dt"], a["g"], a["gdt"], a["A_log"],
                             a["dt_bias"], a["mode"], a["lb"], a["beta"], a["h0"], a["hT"],
                             a["cu"], a["n"], a["B"], a["T"], a["H"], a["K"], a["V"], a["C"],
                             a["o"], a["odt"], a["ws"], a["ws_bytes"], None)


def test_chunk_host_validation(lib):
    assert _chunk(lib, C=48) == UNSUPPORTED
    assert _chunk(lib, K=96) == UNSUPPORTED
    assert _chunk(lib, dt=7) == UNSUPPORTED
    assert _chunk(lib, dt=F32, odt=BF16) == UNSUPPORTED  # float32 inputs write float32 o
    assert _chunk(lib, lb=-5.5) == INVALID
    assert _chunk(lib, lb=0.0) == INVALID
    assert _chunk(lib, A_log=None) == INVALID
    assert _chunk(lib, q=None) == INVALID
    assert _chunk(lib, o=ctypes.c_void_p(4098)) == INVALID  # misaligned
    assert _chunk(lib, B=2, cu=P, n=1) == INVALID  # packed needs B == 1
    # workspace too small (the float32 path needs one; bf16 K=V=128 C=64 needs none)
    assert _chunk(lib, dt=F32, ws=None, ws_bytes=0) == INVALID
    assert b"workspace" in lib.kda_last_error()
    assert _chunk(lib, H=0) == INVALID
    assert _chunk(lib, B=2, T=1 << 30) == INVALID  # B * T reaches 2^31
    assert b"2^31" in lib.kda_last_error()
    # non-safe gate: A_log required, lower_bound ignored, scratch needed for bf16 with
    # K = V = 256 (the stage-by-stage path; K = V = 128 runs the fused kernel without one)
    assert _chunk(lib, mode=2, A_log=None) == INVALID
    assert _chunk(lib, mode=2, lb=0.0, K=256, V=256) == INVALID
    assert b"workspace" in lib.kda_last_error()
    assert _chunk(lib, mode=3) == INVALID
    # nothing to do: zero logical sequences is OK and launches nothing
    assert _chunk(lib, B=0) == OK
    assert _chunk(lib, cu=P, n=0, B=1) == OK


def test_chunk_ex_flags_host_validation(lib):
    """kda_chunk_fwd_ex: unknown option bits are rejected before any launch; with valid bits
    the usual validation still applies first."""
    def ex(flags, **kw):
        a = dict(q=P, o=P, lb=-5.0, C=64, H=2, hk=0)
        a.update(kw)
        return lib.kda_chunk_fwd_ex(a["q"], P, P, BF16, P, BF16, P, None, 1, ctypes.c_float(a["lb"]),
                                    P, None, None, None, 0, 1, 64, a["H"], 128, 128, a["C"], a["o"],
                                    BF16, None, ctypes.c_size_t(0), ctypes.c_int(a["hk"]),
                                    ctypes.c_uint(flags), a.get("status"), None)
    assert ex(2) == INVALID
    assert b"flag" in lib.kda_last_error()
    assert ex(0, H=3, hk=2) == INVALID  # query / key heads must divide the value heads
    assert b"n_qk_heads" in lib.kda_last_error()
    assert ex(0, hk=-1) == INVALID
    assert ex(0x80000000) == INVALID
    assert ex(1, C=48) == UNSUPPORTED
    assert ex(1, q=None) == INVALID
    assert ex(1, lb=0.0) == INVALID
    assert ex(0, status=ctypes.c_void_p(4098)) == INVALID  # the status word must be 4-byte aligned
    assert b"status" in lib.kda_last_error()


def test_recurrent_and_gate_host_validation(lib):
    r = lib.kda_recurrent_fwd(P, P, P, BF16, None, P, None, None, None, 0, 1, 4, 2, 128, 128, P,
                              BF16, None)
    assert r == INVALID  # null gate
    r = lib.kda_recurrent_fwd(P, P, P, BF16, P, P, None, None, None, 0, 1, 4, 2, 300, 128, P, BF16,
                              None)
    assert r == UNSUPPORTED  # K above 256 (any K, V in [1, 256] is accepted)
    r = lib.kda_recurrent_fwd(P, P, P, BF16, P, P, None, None, None, 0, 1, 4, 2, 128, 0, P, BF16,
                              None)
    assert r == UNSUPPORTED

    def rex(mode=3, flags=0, A_log=None, gdt=F32):
        return lib.kda_recurrent_fwd_ex(P, P, P, BF16, P, gdt, A_log, None, mode, ctypes.c_float(-5.0),
                                        P, None, None, None, 0, 1, 4, 2, 128, 128, P, BF16,
                                        ctypes.c_int(0), ctypes.c_uint(flags), None)
    assert rex(flags=8) == INVALID and b"flag" in lib.kda_last_error()
    assert rex(mode=1) == INVALID  # in-kernel gate without A_log
    assert rex(mode=2) == INVALID
    assert rex(mode=4) == INVALID
    assert rex(gdt=7) == UNSUPPORTED
    r = lib.kda_recurrent_fwd_ex(P, P, P, BF16, P, F32, None, None, 3, ctypes.c_float(0.0), P, None,
                                 None, None, 0, 1, 4, 4, 128, 128, P, BF16, ctypes.c_int(3),
                                 ctypes.c_uint(0), None)
    assert r == INVALID  # 3 query / key heads do not divide 4 value heads
    g = lib.kda_gate_fwd(P, BF16, None, None, 1, -5.0, None, 0, 1, 4, 2, 128, 64, P, None)
    assert g == INVALID  # safe gate without A_log
    g = lib.kda_gate_fwd(P, BF16, P, None, 1, -5.0, None, 0, 1, 4, 2, 128, 48, P, None)
    assert g == UNSUPPORTED
    g = lib.kda_gate_fwd(P, BF16, None, None, 2, 0.0, None, 0, 1, 4, 2, 128, 64, P, None)
    assert g == INVALID  # non-safe gate without A_log
    g = lib.kda_gate_fwd(P, BF16, P, None, 3, 0.0, None, 0, 1, 4, 2, 128, 64, P, None)
    assert g == INVALID  # no such mode


def test_launch_counts(lib):
    f = lib.kda_chunk_fwd_launches
    SAFE, NONSAFE = 1, 2
    assert f(F32, F32, 1, 128, 2, 64, 64, 64, 0, SAFE) == 6           # stage-by-stage
    assert f(BF16, BF16, 4, 4096, 64, 256, 256, 64, 0, SAFE) == 2      # two-pass
    assert f(BF16, BF16, 4, 4096, 64, 256, 256, 64, 0, NONSAFE) == 2   # two-pass, non-safe instance
    assert f(BF16, BF16, 4, 4096, 64, 128, 256, 64, 0, SAFE) == 2      # K != V: two-pass
    assert f(BF16, BF16, 4, 4096, 64, 256, 128, 64, 0, NONSAFE) == 2
    assert f(BF16, BF16, 4, 4096, 64, 64, 128, 64, 0, SAFE) == 6       # K = 64: stages
    assert f(BF16, BF16, 4, 4096, 64, 128, 64, 64, 0, SAFE) == 6       # V = 64: stages
    assert f(BF16, BF16, 4, 4096, 64, 128, 128, 64, 0, NONSAFE) == 1   # fused, non-safe instance
    assert f(BF16, BF16, 1, 20480, 32, 128, 128, 32, 16, NONSAFE) == 1
    assert f(BF16, BF16, 1, 20480, 32, 128, 128, 32, 16, SAFE) == 1   # fused, packed
    assert f(BF16, F32, 4, 4096, 64, 128, 128, 64, 0, SAFE) in (1, 2)  # split: by the SM count
    lib.kda_test_hooks(-1, 152, 0, 0)  # plan for 152 SMs: 160 units split in two launches ...
    try:
        assert f(BF16, BF16, 1, 4096, 160, 128, 128, 64, 0, SAFE) == 2
        assert f(BF16, BF16, 1, 4096, 160, 128, 128, 64, 0, NONSAFE) == 1  # ... never the non-safe gate
    finally:
        lib.kda_test_hooks(-1, 0, 0, 0)
    assert f(BF16, BF16, 0, 4096, 64, 128, 128, 64, 0, SAFE) == 0     # no sequences
    assert f(BF16, BF16, 4, 4096, 64, 128, 128, 48, 0, SAFE) == -1    # chunk size
    assert f(BF16, BF16, 4, 4096, 64, 128, 128, 64, 0, 7) == -1       # gate mode
    assert f(BF16, BF16, 2, 4096, 64, 128, 128, 64, 3, SAFE) == -1    # packed needs B == 1
    assert f(F32, BF16, 1, 128, 2, 64, 64, 64, 0, SAFE) == -1         # o dtype


def test_workspace_bytes(lib):
    def al(x):
        return (x + 255) // 256 * 256

    # float32 stage-by-stage path: G, Akk, Aqk, T, w, u, v_new token-indexed + h per chunk slot
    B, T, H, K, V, C = 2, 100, 3, 64, 128, 32
    tt = B * T * H
    slots = B * ((T + C - 1) // C)
    want = sum(al(4 * x) for x in (tt * K, tt * C, tt * C, tt * C, tt * K, tt * V, tt * V,
                                   slots * H * K * V))
    assert lib.kda_chunk_workspace_bytes(F32, B, T, H, K, V, C, 0) == want
    # packed: floor(T_cap / C) + N + 1 chunk slots
    n = 5
    slots = T // C + n + 1
    tt = T * H
    want = sum(al(4 * x) for x in (tt * K, tt * C, tt * C, tt * C, tt * K, tt * V, tt * V,
                                   slots * H * K * V))
    assert lib.kda_chunk_workspace_bytes(F32, 1, T, H, K, V, C, n) == want
    assert lib.kda_chunk_workspace_bytes(F32, 1, T, H, K, V, 48, 0) == 0
    # the fused bf16 kernel keeps every intermediate on chip
    assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 128, 128, 64, 0) == 0
    assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 128, 128, 32, 0) == 0  # fused too
    # the two-pass path (K = V = 256): per 64-token chunk and head, T diag(beta) bf16 and Aqk fp32
    # (24 KB), k 2^G, s q 2^G and k 2^(Gl - G) in bf16 (3 x 64 K 2 bytes), 2^Glast (K floats) and
    # the q^2 row sums (64 floats)
    def img(K):
        return 24576 + 3 * 64 * K * 2 + 4 * K + 256

    assert img(256) == 124160 and img(128) == 74496
    lib.kda_test_hooks(-1, 0, 1, 0)  # one CTA per unit in pass 2 (no balanced schedule)
    try:
        assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 256, 256, 64, 0) == 4 * 64 * 64 * img(256)
        assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 256, 256, 32, 0) == 4 * 64 * 64 * img(256)
    finally:
        lib.kda_test_hooks(-1, 0, 0, 0)
    # packed: floor(T_cap / 64) + N + 1 chunk slots
    assert lib.kda_chunk_workspace_bytes(BF16, 1, 20480, 32, 256, 256, 64, 16) == (320 + 17) * 32 * img(256)
    # the two-pass test hook moves K = V = 128 onto it
    lib.kda_test_hooks(-1, 0, 1, 1)
    try:
        assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 128, 128, 64, 0) == 4 * 64 * 64 * img(128)
        assert lib.kda_chunk_fwd_launches(BF16, BF16, 4, 4096, 64, 128, 128, 64, 0, 1) == 2
    finally:
        lib.kda_test_hooks(-1, 0, 0, 0)
    assert lib.kda_chunk_workspace_bytes(BF16, 4, 4096, 64, 128, 128, 64, 0) == 0
    # by gate mode: the fused and two-pass kernels take every mode; float32 inputs and head dims
    # of 64 run on the stage-by-stage path
    ex = lib.kda_chunk_workspace_bytes_ex
    ex.restype = ctypes.c_size_t
    assert ex(BF16, 4, 4096, 64, 128, 128, 64, 0, 0) == 0
    assert ex(BF16, 4, 4096, 64, 128, 128, 64, 0, 1) == 0
    assert ex(BF16, 4, 4096, 64, 128, 128, 64, 0, 2) == 0
    assert ex(BF16, 4, 2048, 8, 256, 256, 64, 0, 2) == 4 * 32 * 8 * img(256)  # 32 units: one wave
    assert ex(F32, 4, 2048, 8, 256, 256, 64, 0, 2) == lib.kda_chunk_workspace_bytes(
        F32, 4, 2048, 8, 256, 256, 64, 0) > 0
    assert ex(BF16, 4, 4096, 64, 128, 128, 64, 0, 3) == 0  # no such mode
    assert ex(F32, B, T, H, K, V, C, 0, 2) == lib.kda_chunk_workspace_bytes(F32, B, T, H, K, V, C, 0)


def test_split_schedule_plan(lib):
    """The two-launch plan for dense fused calls, on a stated SM count (no device needed): it
    splits only when the last wave of (sequence, head) units is at most half full and the second
    pieces hold the FP32 state in their output rows (256 bf16 rows, 128 float32 rows)."""
    f = lib.kda_chunk_fwd_launches
    SAFE = 1

    def launches(B, T, H, o=BF16, S=152):
        lib.kda_test_hooks(-1, S, 0, 0)
        return f(BF16, o, B, T, H, 128, 128, 64, 0, SAFE)

    assert launches(2, 720, 114) == 2        # 228 units: the last wave half full
    assert launches(1, 4096, 160) == 2       # 160 units: 8 in the last wave
    assert launches(1, 8192, 200) == 2
    assert launches(4, 4096, 64) == 1        # 256 units: 68 % full, four rounds of pieces
    assert launches(1, 4096, 152) == 1       # whole waves
    assert launches(1, 4096, 304) == 1
    assert launches(1, 4096, 100) == 1       # fewer units than SMs
    assert launches(2, 320, 114) == 1        # 5 chunks: the second pieces too short
    assert launches(2, 512, 114) == 1        # 192-token second pieces: too short for bf16 o ...
    assert launches(2, 512, 114, o=F32) == 2  # ... long enough for a float32 o
    assert launches(1, 4096, 12, S=8) == 2   # any SM count
    assert launches(1, 20480, 32, S=8) == 1  # a whole number of waves
    assert f(BF16, BF16, 1, 4096, 160, 128, 128, 64, 3, SAFE) == 1  # packed: never split
    lib.kda_test_hooks(-1, 152, 1, 0)  # one launch whatever the plan
    assert f(BF16, BF16, 2, 720, 114, 128, 128, 64, 0, SAFE) == 1
    lib.kda_test_hooks(-1, 0, 0, 0)  # hooks off again


def test_two_pass_balanced_plan(lib):
    """Pass 2's balanced schedule, on a stated SM count S (no device needed): dense inputs whose
    N H units leave the last wave of a one-CTA-per-unit grid part-empty on S / (V / 128) groups
    of SMs, where ceil(U nt / groups) + 2 chunk-times beat it by 5 % or more.  It adds one flag
    per CTA (rounded to 256 bytes) and one FP32 K x 128 state slot per CTA to the workspace; the
    call still makes two launches."""
    img = 124160  # K = 256 image bytes per chunk and head

    def ws(B, T, H, V=256, S=152, mode=1, n=0):
        lib.kda_test_hooks(-1, S, 0, 0)
        assert lib.kda_chunk_fwd_launches(BF16, BF16, B, T, H, 256, V, 64, n, mode) == 2
        return lib.kda_chunk_workspace_bytes_ex(BF16, B, T, H, 256, V, 64, n, mode)

    def bal(S, V=256):
        slots = S // (V // 128) * (V // 128)
        return (slots * 4 + 255) // 256 * 256 + slots * 256 * 128 * 4

    try:
        base = 8 * 32 * 32 * img
        assert ws(8, 2048, 32) == base + bal(152)          # 256 units on 76 groups: 108 against 128
        assert ws(8, 2048, 32, mode=2) == base + bal(152)  # the non-safe gate too
        assert ws(8, 2048, 32, S=151) == base + bal(151)   # 75 groups of two
        assert ws(4, 1000, 40) == 4 * 16 * 40 * img + bal(152)
        assert ws(2, 2048, 38) == 2 * 32 * 38 * img        # 76 units: one whole wave
        assert ws(1, 2048, 60) == 32 * 60 * img            # fewer units than groups
        assert ws(4, 2048, 57) == 4 * 32 * 57 * img        # 228 units = 3 waves
        assert ws(1, 20480, 32, n=3) == (320 + 4) * 32 * img  # packed: never
        lib.kda_test_hooks(-1, 152, 1, 0)  # one CTA per unit whatever the plan
        assert lib.kda_chunk_workspace_bytes(BF16, 8, 2048, 32, 256, 256, 64, 0) == base
    finally:
        lib.kda_test_hooks(-1, 0, 0, 0)


def test_no_environment_hooks():
    """The library reads no environment variables: its test hooks are set only through
    kda_test_hooks."""
    for src in os.listdir(os.path.join(ROOT, "chunked_kda_gb300", "csrc")):
        text = open(os.path.join(ROOT, "chunked_kda_gb300", "csrc", src)).read()
        assert "getenv" not in text, src


def test_layout_and_alignment_validation(lib):
    """The remaining host checks of the layout, the packed offsets, the workspace and the gate
    entry point: each is reported before any launch."""
    assert _chunk(lib, B=1, T=1 << 30, H=1 << 11) == INVALID  # more than 2^40 elements
    assert b"too large" in lib.kda_last_error()
    assert _chunk(lib, B=65536, T=1) == INVALID
    assert b"65535" in lib.kda_last_error()
    assert _chunk(lib, cu=P, n=65536, B=1) == INVALID
    assert _chunk(lib, cu=ctypes.c_void_p(4098), n=2, B=1) == INVALID
    assert b"misaligned" in lib.kda_last_error()
    need = lib.kda_chunk_workspace_bytes(F32, 1, 64, 2, 128, 128, 64, 0)
    assert need > 0
    assert _chunk(lib, dt=F32, gdt=F32, ws=ctypes.c_void_p(4096 + 16), ws_bytes=need) == INVALID
    assert b"256-byte" in lib.kda_last_error()
    assert lib.kda_gate_fwd(None, BF16, P, None, 1, -5.0, None, 0, 1, 4, 2, 128, 64, P, None) == INVALID
    assert lib.kda_gate_fwd(P, BF16, P, None, 1, -5.0, None, 0, 1, 4, 2, 128, 64, None, None) == INVALID
    assert b"null g" in lib.kda_last_error()
    assert lib.kda_gate_fwd(P, BF16, P, None, 1, -5.0, None, 0, 1, 4, 2, 0, 64, P, None) == INVALID


def _noalloc(lib, **kw):
    a = dict(q=P, k=P, v=P, dt=F32, g=P, gdt=F32, A_log=P, dt_bias=None, mode=1, lb=-5.0,
             beta=P, h0=None, hT=None, cu=None, n=0, B=1, T=64, H=2, K=128, V=128, C=64, o=P,
             odt=None)
    a.update(kw)
    if a["odt"] is None:
        a["odt"] = a["dt"]
    return lib.kda_chunk_fwd_noalloc(a["q"], a["k"], a["v"], a["dt"], a["g"], a["gdt"], a["A_log"],
                                     a["dt_bias"], a["mode"], a["lb"], a["beta"], a["h0"], a["hT"],
                                     a["cu"], a["n"], a["B"], a["T"], a["H"], a["K"], a["V"], a["C"],
                                     a["o"], a["odt"], None)


def test_noalloc_host_validation_is_kda_chunk_fwds(lib):
    """kda_chunk_fwd_noalloc runs kda_chunk_fwd's host checks, size limits included, before
    it looks anything up on the device."""
    assert _noalloc(lib, C=48) == UNSUPPORTED
    assert _noalloc(lib, K=96) == UNSUPPORTED
    assert _noalloc(lib, dt=F32, odt=BF16) == UNSUPPORTED
    assert _noalloc(lib, lb=0.0) == INVALID
    assert _noalloc(lib, A_log=None) == INVALID
    assert _noalloc(lib, q=None) == INVALID
    assert _noalloc(lib, o=ctypes.c_void_p(4098)) == INVALID
    assert _noalloc(lib, B=2, cu=P, n=1) == INVALID
    assert _noalloc(lib, cu=ctypes.c_void_p(4098), n=1) == INVALID  # misaligned offsets
    # B * T must stay below 2^31 (token coordinates are 32-bit), B * T * H at most 2^40
    assert _noalloc(lib, B=2, T=1 << 30) == INVALID
    assert b"2^31" in lib.kda_last_error()
    assert _noalloc(lib, B=1, T=(1 << 31) - 1, H=1 << 10) == INVALID
    # a size far beyond the fixed scratch is refused before any device work
    assert _noalloc(lib, B=1, T=1 << 20, H=8) == INVALID
    assert b"KDA_NOALLOC_SCRATCH_BYTES" in lib.kda_last_error()
    # no sequences: nothing to do
    assert _noalloc(lib, B=0) == OK
