"""C-ABI checks that need no GPU: build, load, exported symbols, struct layout,
host-side argument validation.  No call here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cgdr.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cg.lib()


def declared_functions(headers=None):
    names = set()
    for h in headers or HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(cgdr_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_abi():
    assert declared_functions([HEADER]) == sorted([
        "cgdr_abi_version", "cgdr_status_string", "cgdr_validate", "cgdr_decode",
        "cgdr_prefill_workspace_size", "cgdr_prefill", "cgdr_workspace_status", "cgdr_prefill_noalloc",
        "cgdr_prefill_path_for"])
    assert declared_functions([os.path.join(ROOT, "include", "cgdr_debug.h")]) == ["cgdr_debug_decode_shrunk_o"]


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return set(re.findall(r"\b[TW] (\w+)$", out, flags=re.M))


def test_library_exports_every_declared_symbol(lib):
    exported = _exports(cg.LIB_PATH)
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_debug_library_builds_and_exports_every_declared_symbol():
    """The index-checking build compiles from the same sources and exports the same ABI plus
    its test entry point; the release library answers that entry point with UNSUPPORTED."""
    path = cbuild.build(debug=True)
    exported = _exports(path)
    for name in declared_functions():
        assert name in exported, name
    dlib = ctypes.CDLL(path)
    dlib.cgdr_abi_version.restype = ctypes.c_int
    assert dlib.cgdr_abi_version() == cg.lib().cgdr_abi_version()
    rel = cg.lib()
    rel.cgdr_debug_decode_shrunk_o.restype = ctypes.c_int
    rel.cgdr_debug_decode_shrunk_o.argtypes = [ctypes.POINTER(cg.CgdrArgs), ctypes.c_int64, ctypes.c_void_p]
    A = _args()
    assert rel.cgdr_debug_decode_shrunk_o(ctypes.byref(A), 4, None) == cg.ERR_UNSUPPORTED


def test_abi_version_and_status_strings(lib):
    m = re.search(r"#define CGDR_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.cgdr_abi_version() == int(m.group(1))
    for s in range(9):
        assert cg.status_string(s).startswith("CGDR_")
    assert cg.status_string(99) == "unknown cgdr status"


def test_struct_layout_matches_c(tmp_path):
    """ctypes mirror of cgdr_args has the size and field offsets the C compiler gives."""
    fields = [f[0] for f in cg.CgdrArgs._fields_]
    src = tmp_path / "layout.c"
    body = "\n".join('printf("%s %%zu\\n", offsetof(cgdr_args, %s));' % (f, f) for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "cgdr.h"\nint main(void){\n'
                   'printf("sizeof %zu\\n", sizeof(cgdr_args));\n' + body + "\nreturn 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n") if l)
    assert int(got["sizeof"]) == ctypes.sizeof(cg.CgdrArgs)
    for f in fields:
        assert int(got[f]) == getattr(cg.CgdrArgs, f).offset, f


def _args(**kw):
    """A valid-looking bf16 channel-gate argument block with fake (never dereferenced) pointers."""
    A = cg.CgdrArgs()
    A.B, A.T, A.Hk, A.Hv, A.dk, A.dv = 2, 1, 2, 4, 128, 128
    A.dtype, A.gate, A.l2norm_qk, A.chunk = cg.BF16, cg.GATE_CHANNEL, 1, 64
    base = 1 << 20
    for i, name in enumerate(["q", "k", "v", "o", "g", "beta", "state"]):
        setattr(A, name, base * (i + 1))
    A.q_sb, A.q_st, A.q_sh = 8 * 128, 2 * 128, 128
    A.k_sb, A.k_st, A.k_sh = 8 * 128, 2 * 128, 128
    A.v_sb, A.v_st, A.v_sh = 16 * 128, 4 * 128, 128
    A.o_sb, A.o_st, A.o_sh = 16 * 128, 4 * 128, 128
    A.g_sb, A.g_st, A.g_sh = 16 * 128, 4 * 128, 128
    A.beta_sb, A.beta_st, A.beta_sh = 4, 4, 1
    for k, v in kw.items():
        setattr(A, k, v)
    return A


def test_validation_accepts_good_args(lib):
    assert cg.validate(_args(), False) == cg.OK
    assert cg.validate(_args(T=5), True) == cg.OK


@pytest.mark.parametrize("kw,prefill,code", [
    (dict(T=2), False, cg.ERR_INVALID_ARG),            # decode is T == 1
    (dict(Hv=3), False, cg.ERR_INVALID_ARG),           # Hv % Hk
    (dict(B=-1), False, cg.ERR_INVALID_ARG),
    (dict(Hk=0), True, cg.ERR_INVALID_ARG),
    (dict(q=0), False, cg.ERR_INVALID_ARG),
    (dict(state=0), True, cg.ERR_INVALID_ARG),
    (dict(g=0), False, cg.ERR_INVALID_ARG),
    (dict(gate=cg.GATE_GDN), False, cg.ERR_INVALID_ARG),  # a, b, A_log, dt_bias missing
    (dict(dk=96), False, cg.ERR_UNSUPPORTED),
    (dict(dv=256), True, cg.ERR_UNSUPPORTED),
    (dict(dtype=7), False, cg.ERR_UNSUPPORTED),
    (dict(gate=5), False, cg.ERR_UNSUPPORTED),
    (dict(chunk=48), True, cg.ERR_UNSUPPORTED),
    (dict(o_dtype=3), False, cg.ERR_UNSUPPORTED),
    (dict(o_dtype=cg.BF16, o_sh=132), False, cg.ERR_ALIGNMENT),   # bf16 o: strides of 8 elements
    (dict(q=(1 << 20) + 2), False, cg.ERR_ALIGNMENT),
    (dict(state=(7 << 20) + 4), False, cg.ERR_ALIGNMENT),
    (dict(q_sh=100), False, cg.ERR_ALIGNMENT),
    (dict(v_st=12), True, cg.ERR_ALIGNMENT),
    (dict(g_sb=2), False, cg.ERR_ALIGNMENT),
    (dict(o_sb=-8), False, cg.ERR_ALIGNMENT),
    (dict(prefill_path=6), True, cg.ERR_INVALID_ARG),
    (dict(prefill_path=-1), True, cg.ERR_INVALID_ARG),
    (dict(status=(9 << 20) + 2), False, cg.ERR_ALIGNMENT),
])
def test_validation_rejects(lib, kw, prefill, code):
    A = _args(**kw)
    assert cg.validate(A, prefill) == code
    # the entry points return the same code without touching the GPU
    if prefill:
        assert lib.cgdr_prefill(ctypes.byref(A), None, 0, None) == code
        assert lib.cgdr_prefill_workspace_size(ctypes.byref(A)) == 0
    else:
        assert lib.cgdr_decode(ctypes.byref(A), None) == code


def test_empty_work_is_a_no_op(lib):
    # B == 0 or T == 0: nothing to do, pointers may be NULL, no launch happens
    A = _args(B=0, q=0, k=0, v=0, o=0, g=0, beta=0, state=0)
    assert lib.cgdr_decode(ctypes.byref(A), None) == cg.OK
    A = _args(T=0, q=0, k=0, v=0, o=0, g=0, beta=0, state=0)
    assert lib.cgdr_prefill(ctypes.byref(A), None, 0, None) == cg.OK
    assert lib.cgdr_validate(None, 0) == cg.ERR_INVALID_ARG


def test_workspace_rules(lib):
    A = _args(T=100)
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(A)) == 256     # tensor-core path: error word
    assert lib.cgdr_prefill(ctypes.byref(A), None, 0, None) == cg.ERR_WORKSPACE
    assert lib.cgdr_prefill(ctypes.byref(A), ctypes.c_void_p(1 << 30), 64, None) == cg.ERR_WORKSPACE
    assert lib.cgdr_prefill(ctypes.byref(A), ctypes.c_void_p((1 << 30) + 4), 256, None) == cg.ERR_WORKSPACE
    A32 = _args(T=100, dtype=cg.F32, q_sb=8 * 128, q_st=2 * 128, q_sh=128)
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(A32)) == 0      # fp32 inputs: CUDA-core path
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(_args(T=100, chunk=32))) == 0
    assert lib.cgdr_workspace_status(None, None) == cg.ERR_INVALID_ARG


def test_wait_polls_values_are_accepted(lib):
    # 0: default limit; > 0: that many polls; < 0: the injected-failure test hook
    for polls in (0, 1, 1000, -1, -(1 << 31)):
        assert cg.validate(_args(wait_polls=polls), False) == cg.OK


def test_output_dtype_strides(lib):
    assert cg.validate(_args(o_dtype=cg.F32, o_sh=132), False) == cg.OK     # fp32 o: 4-element strides
    assert cg.validate(_args(o_dtype=cg.BF16, o_sh=136), False) == cg.OK


def test_token_strides_ignored_by_decode(lib):
    assert cg.validate(_args(q_st=3, v_st=5, o_st=1, g_st=7), False) == cg.OK


def test_prefill_path_choice(lib):
    """Kernel selection is host logic, taken from the call's own argument block: a forced
    tensor-core kernel applies only to the shapes it covers (bf16, dk = dv = 128, chunk 64);
    out-of-range choices are rejected."""
    path_for = lambda A: lib.cgdr_prefill_path_for(ctypes.byref(A))
    for bad in (6, -1, 9):
        assert path_for(_args(T=100, prefill_path=bad)) == cg.PREFILL_AUTO       # invalid arguments
    for path in (cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_SIMT):
        assert path_for(_args(T=100, prefill_path=path)) == path
        for other in (dict(T=100, chunk=32), dict(T=100, dv=64),
                      dict(T=100, dtype=cg.F32, q_sb=8 * 128, q_st=2 * 128, q_sh=128)):
            assert path_for(_args(prefill_path=path, **other)) == cg.PREFILL_SIMT
    # 1 <= T <= 8: the token recurrence under the automatic choice (or when forced); a forced
    # chunked kernel still runs chunked; RECURRENT forced on a longer T means the automatic choice
    for T in (1, 2, 8):
        for kw in ({}, dict(dtype=cg.F32, q_sb=8 * 128, q_st=2 * 128, q_sh=128), dict(dk=32, dv=64)):
            assert path_for(_args(T=T, **kw)) == cg.PREFILL_RECURRENT
        assert lib.cgdr_prefill_workspace_size(ctypes.byref(_args(T=T))) == 0
    assert path_for(_args(T=9)) in (cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP)
    assert path_for(_args(T=2, prefill_path=cg.PREFILL_PER_HEAD)) == cg.PREFILL_PER_HEAD
    assert path_for(_args(T=3, prefill_path=cg.PREFILL_RECURRENT)) == cg.PREFILL_RECURRENT
    assert path_for(_args(T=100, prefill_path=cg.PREFILL_RECURRENT)) in (cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER,
                                                                         cg.PREFILL_COOP)
    # the cooperative kernel needs more resident CTAs than heads; without a device it falls back
    assert path_for(_args(T=100, prefill_path=cg.PREFILL_COOP)) in (cg.PREFILL_COOP, cg.PREFILL_PER_HEAD,
                                                                    cg.PREFILL_CLUSTER)
    assert path_for(_args(T=0)) == cg.PREFILL_AUTO
    assert path_for(_args(T=100, dk=96)) == cg.PREFILL_AUTO
    assert lib.cgdr_prefill_path_for(None) == cg.PREFILL_AUTO
    # workspace by kernel: status word; status word + nine hand-off slots per (batch, v-head)
    A = _args(T=100, prefill_path=cg.PREFILL_PER_HEAD)
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(A)) == 256
    A = _args(T=100, prefill_path=cg.PREFILL_CLUSTER)
    need = 256 + A.B * A.Hv * 9 * 82432
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(A)) == need
    assert lib.cgdr_prefill(ctypes.byref(A), None, 0, None) == cg.ERR_WORKSPACE
    assert lib.cgdr_prefill(ctypes.byref(A), ctypes.c_void_p(1 << 30), need - 16, None) == cg.ERR_WORKSPACE
    assert lib.cgdr_prefill_workspace_size(ctypes.byref(_args(T=100, prefill_path=cg.PREFILL_SIMT))) == 0


def test_calls_from_two_threads_do_not_interfere(lib):
    """The kernel choice lives in each call's argument block: two host threads asking for
    different kernels (and their workspace sizes) at the same time each get their own answer."""
    import threading
    errors = []

    def worker(path, expect_ws):
        A = _args(T=100, prefill_path=path)
        for _ in range(2000):
            if lib.cgdr_prefill_path_for(ctypes.byref(A)) != path or \
                    lib.cgdr_prefill_workspace_size(ctypes.byref(A)) != expect_ws:
                errors.append(path)
                return

    ts = [threading.Thread(target=worker, args=(cg.PREFILL_PER_HEAD, 256)),
          threading.Thread(target=worker, args=(cg.PREFILL_CLUSTER, 256 + 2 * 4 * 9 * 82432)),
          threading.Thread(target=worker, args=(cg.PREFILL_SIMT, 0))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors


def test_tensor_maps_cover_strides_or_fall_back(lib):
    """The tensor-core prefill stages rows with TMA tensor maps; strides a map cannot take
    (a zero or negative stride over an extent above one, or one of 2^40 bytes or more) send
    the call to the CUDA-core kernel, and a dimension of extent one may carry any stride."""
    P = cg.PREFILL_PER_HEAD
    path_for = lambda **kw: lib.cgdr_prefill_path_for(ctypes.byref(_args(prefill_path=P, **kw)))
    assert path_for(T=100) == P
    # q heads sharing one row (head stride 0) with Hk = 2: valid input, no tensor map
    assert cg.validate(_args(T=100, q_sh=0), True) == cg.OK
    assert path_for(T=100, q_sh=0) == cg.PREFILL_SIMT
    # a batch stride of 2^40 bytes and more (bf16: 2^39 elements)
    assert path_for(T=100, k_sb=1 << 39) == cg.PREFILL_SIMT
    # extent-one dimensions: their strides never step, so any value is fine
    one = dict(T=100, B=1, Hk=1, Hv=1)
    for kw in (dict(q_sh=0, k_sh=0, v_sh=0, g_sh=0), dict(q_sb=0, k_sb=0, v_sb=0, g_sb=0)):
        assert path_for(**one, **kw) == P
