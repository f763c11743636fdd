"""CPU checks of the C ABI: the library builds, loads, and exports every function that
include/gqmm.h declares; argument validation rejects bad calls before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gqmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(gqmm_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from quantized_moe_expert_device_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gqmm_quantize", "gqmm_route_sort", "gqmm_gather_qmm", "gqmm_workspace_size",
                     "gqmm_device_status", "gqmm_status_string"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gqmm.h but not exported"


def test_binding_covers_the_boundary():
    import quantized_moe_expert_device_gb300 as g

    lib = g.load_library()
    for name in ("gqmm_quantize", "gqmm_route_sort", "gqmm_gather_qmm", "gqmm_workspace_size",
                 "gqmm_device_status", "gqmm_gather_qmm_simt", "gqmm_moe_mlp", "gqmm_moe_mlp_workspace_size",
                 "gqmm_gather_qmm_nn", "gqmm_gather_qmm_nn_simt"):
        assert hasattr(g, name)
        assert getattr(lib, name).argtypes is not None


def test_workspace_size_is_positive_and_monotone(lib):
    import quantized_moe_expert_device_gb300 as g

    # above the split-K size limit the workspace grows with the number of rows
    a = g.gqmm_workspace_size(2048, 768, 64)
    b = g.gqmm_workspace_size(16384, 768, 64)
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0
    # a decode-sized call (9 work units at most) has room for 16 split-K float32 planes
    c = g.gqmm_workspace_size(32, 128, 8)
    assert c % 256 == 0 and c >= 16 * 32 * 128 * 4
    assert g.gqmm_workspace_size(10, 128, 0) == 0
    assert g.gqmm_workspace_size(10, 128, 4096) == 0


def test_validation_rejects_bad_arguments_without_a_gpu(lib):
    # Validation runs before any CUDA call, so these return codes are exact on any host.
    P = ctypes.c_void_p
    f = lib.gqmm_gather_qmm
    f.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    args = dict(x=fake, wq=fake, sc=fake, bs=fake, idx=fake, T=16, A=2, H=256, F=128, E=8, gs=64, bits=4,
                sorted=0, shared=0, y=fake, ws=fake, wsb=1 << 20, s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["x"], a["wq"], a["sc"], a["bs"], a["idx"], a["T"], a["A"], a["H"], a["F"], a["E"], a["gs"],
                 a["bits"], a["sorted"], a["shared"], a["y"], a["ws"], a["wsb"], a["s"])

    assert call(x=None) == 1                  # ERR_NULL
    assert call(shared=2) == 2                # x_shared is 0 or 1
    assert call(shared=1, idx=None, E=1) == 1  # a shared x needs the routed rows of idx
    assert call(gs=96) == 3                   # ERR_UNSUPPORTED: group sizes are 32, 64 and 128
    assert call(gs=16) == 3
    assert call(gs=256) == 3
    assert call(gs=128, H=192) == 2           # ERR_SHAPE: H must be a multiple of the group size
    assert call(bits=7) == 3                  # code widths are 2, 3, 4, 5, 6 and 8
    assert call(bits=8, gs=128) == 3          # widths other than 4 take 64-wide groups only
    assert call(bits=3, H=192) == 2           # a row's 3-bit codes (72 bytes) are no multiple of 16 bytes
    assert call(H=100) == 2                   # ERR_SHAPE
    assert call(F=120) == 2
    assert call(T=0) == 2
    assert call(E=0) == 2
    assert call(E=4096) == 3
    assert call(idx=None) == 1                # dense needs E == 1
    assert call(x=P(0x10008)) == 4            # ERR_ALIGN
    assert call(sorted=2) == 2
    assert call(wsb=16) == 5                  # ERR_WORKSPACE
    lib.gqmm_last_error.restype = ctypes.c_char_p
    assert b"workspace" in lib.gqmm_last_error()
    lib.gqmm_status_string.restype = ctypes.c_char_p
    assert lib.gqmm_status_string(0) == b"ok"


def test_mlp_validation_rejects_bad_arguments_without_a_gpu(lib):
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f = lib.gqmm_moe_mlp
    f.argtypes = [P, P, P, P, P, P, P, P, I64, I, I, I, I, I, I, I, I, I, P, P, ctypes.c_size_t, P]
    f.restype = I
    lib.gqmm_moe_mlp_workspace_size.argtypes = [I64, I, I, I]
    lib.gqmm_moe_mlp_workspace_size.restype = ctypes.c_size_t
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    args = dict(x=fake, wgu=fake, sgu=fake, bgu=fake, wdn=fake, sdn=fake, bdn=fake, idx=fake, T=16, A=2, H=256,
                I=128, E=8, gs=64, bits=4, act=0, sorted=0, shared=0, y=fake, ws=fake, wsb=1 << 20, s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["x"], a["wgu"], a["sgu"], a["bgu"], a["wdn"], a["sdn"], a["bdn"], a["idx"], a["T"], a["A"],
                 a["H"], a["I"], a["E"], a["gs"], a["bits"], a["act"], a["sorted"], a["shared"], a["y"], a["ws"],
                 a["wsb"], a["s"])

    assert call(wdn=None) == 1                # ERR_NULL (down projection)
    assert call(x=None) == 1
    assert call(I=96) == 2                    # ERR_SHAPE: I is the down projection's K (multiple of 64)
    assert call(I=0) == 2
    assert call(H=100) == 2
    assert call(gs=96) == 3                   # ERR_UNSUPPORTED
    assert call(gs=128, I=192) == 2           # ERR_SHAPE: I (the down projection's K) % group_size
    assert call(act=3) == 3                   # no such activation
    assert call(shared=3) == 2
    assert call(act=-1) == 3
    assert call(idx=None) == 1                # dense needs E == 1
    assert call(sorted=3) == 2
    assert call(wsb=16) == 5                  # ERR_WORKSPACE
    assert lib.gqmm_moe_mlp_workspace_size(32, 256, 128, 8) > lib.gqmm_moe_mlp_workspace_size(32, 256, 64, 8) > 0
    assert lib.gqmm_moe_mlp_workspace_size(32, 256, 0, 8) == 0
    assert lib.gqmm_moe_mlp_workspace_size(32, 256, 128, 0) == 0


def test_nn_validation_rejects_bad_arguments_without_a_gpu(lib):
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    f = lib.gqmm_gather_qmm_nn
    f.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I, I, I, P, P, SZ, P]
    f.restype = I
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    args = dict(x=fake, wq=fake, sc=fake, bs=fake, idx=fake, T=16, A=2, K=256, N=128, E=8, gs=64, bits=4, sorted=0,
                shared=0, y=fake, ws=fake, wsb=1 << 30, s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["x"], a["wq"], a["sc"], a["bs"], a["idx"], a["T"], a["A"], a["K"], a["N"], a["E"], a["gs"],
                 a["bits"], a["sorted"], a["shared"], a["y"], a["ws"], a["wsb"], a["s"])

    assert call(wq=None) == 1                 # ERR_NULL
    assert call(gs=96) == 3                   # ERR_UNSUPPORTED
    assert call(bits=2) == 3
    assert call(N=96) == 2                    # ERR_SHAPE: N must be a multiple of the group size
    assert call(N=48, gs=32) == 2             # and of 32 (a code row fills whole 16-byte units)
    assert call(K=0) == 2
    assert call(K=300) == 2                   # K a multiple of the 64-wide k-block
    assert call(T=0) == 2
    assert call(E=0) == 2
    assert call(E=2048) == 3
    assert call(idx=None) == 1                # dense needs E == 1
    assert call(shared=2) == 2
    assert call(shared=1, idx=None, E=1) == 1
    assert call(sorted=2) == 2
    assert call(y=P(0x10008)) == 4            # ERR_ALIGN: y is stored 16 bytes at a time
    assert call(x=P(0x10008)) == 4            # x rows are copied by TMA
    assert call(wq=P(0x10004)) == 4
    assert call(ws=None) == 1
    assert call(wsb=16) == 5                  # ERR_WORKSPACE


def test_nn_simt_validation_rejects_bad_arguments_without_a_gpu(lib):
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f = lib.gqmm_gather_qmm_nn_simt
    f.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P]
    f.restype = I
    fake = P(0x10000)
    args = dict(x=fake, wq=fake, sc=fake, bs=fake, idx=fake, T=16, A=2, K=300, N=128, E=8, gs=64, bits=4, shared=0,
                y=fake, s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["x"], a["wq"], a["sc"], a["bs"], a["idx"], a["T"], a["A"], a["K"], a["N"], a["E"], a["gs"],
                 a["bits"], a["shared"], a["y"], a["s"])

    assert call(wq=None) == 1
    assert call(gs=96) == 3
    assert call(N=96) == 2
    assert call(K=0) == 2
    assert call(idx=None) == 1
    assert call(y=P(0x10008)) == 4


def test_fp_mode_validation_rejects_bad_arguments_without_a_gpu(lib):
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f = lib.gqmm_gather_qmm_fp
    f.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P, ctypes.c_size_t, P]
    f.restype = I
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails before any launch
    args = dict(x=fake, wq=fake, sc=fake, ts=fake, idx=fake, T=16, A=2, H=256, F=128, E=8, mode=1, sorted=0, shared=0,
                y=fake, ws=fake, wsb=1 << 20, s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["x"], a["wq"], a["sc"], a["ts"], a["idx"], a["T"], a["A"], a["H"], a["F"], a["E"], a["mode"],
                 a["sorted"], a["shared"], a["y"], a["ws"], a["wsb"], a["s"])

    assert call(mode=0) == 3 and call(mode=4) == 3  # ERR_UNSUPPORTED: modes 1 (mxfp4), 2 (nvfp4), 3 (mxfp8)
    assert call(sc=None) == 1                        # ERR_NULL
    assert call(mode=2, ts=None) == 1                # nvfp4 needs its per-expert scales
    assert call(H=96) == 2                           # ERR_SHAPE: H a multiple of 64
    assert call(F=24) == 2
    assert call(sc=ctypes.c_void_p((1 << 20) + 2)) == 4  # ERR_ALIGN: scales 4-byte aligned
    assert call(wsb=16) == 5                         # ERR_WORKSPACE

    q = lib.gqmm_quantize_fp
    q.argtypes = [P, I64, I64, I64, I, P, P, P, P]
    q.restype = I
    assert q(fake, 8, 256, 8, 5, fake, fake, fake, None) == 3   # unknown mode
    assert q(fake, 8, 100, 8, 1, fake, fake, None, None) == 2   # H a multiple of 64
    assert q(fake, 8, 256, 3, 2, fake, fake, fake, None) == 2   # nvfp4: rows a multiple of rows_per_tensor
    assert q(fake, 8, 256, 8, 2, fake, fake, None, None) == 1   # nvfp4 needs tscale


def declared_prototypes():
    """name -> (return type, [parameter types]) for every GQMM_API function of gqmm.h, types with
    qualifiers and parameter names stripped (e.g. "void*", "int64_t", "gqmm_stream_t")."""
    text = open(os.path.join(ROOT, "include", "gqmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for ret, name, params in re.findall(r"GQMM_API\s+([\w \*]+?)\s*\b(gqmm_\w+)\s*\(([^)]*)\)\s*;", text):
        types = []
        for prm in [q.strip() for q in params.split(",") if q.strip() and q.strip() != "void"]:
            prm = re.sub(r"\bconst\b", "", prm)
            stars = prm.count("*")
            words = prm.replace("*", " ").split()
            base = words[0] if stars or len(words) == 1 else " ".join(words[:-1])
            types.append(base + "*" * stars)
        protos[name] = (re.sub(r"\bconst\b", "", ret).replace(" ", ""), types)
    return protos


def _ctype_of(c_type):
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    table = {"int": I, "int64_t": I64, "size_t": SZ, "gqmm_stream_t": P, "void": None, "char*": ctypes.c_char_p,
             "int64_t*": ctypes.POINTER(I64), "double*": ctypes.POINTER(ctypes.c_double)}
    if c_type in table:
        return table[c_type]
    assert c_type.endswith("*"), f"unmapped C type {c_type}"
    return P  # data pointers (void*, uint32_t*, int32_t*, float*) travel as void*


def test_binding_signatures_match_the_header():
    """Every function the binding declares to ctypes has the header's parameter count and types
    (an int where the C side takes int64_t, or a missing stream argument, would be undefined
    behaviour at the call), and the header's return type."""
    import quantized_moe_expert_device_gb300 as g

    protos = declared_prototypes()
    assert set(declared_functions()) == set(protos), "every declaration parsed"
    lib = g.load_library()
    checked = 0
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:  # not marshalled by the binding (called directly through ctypes)
            continue
        want = [_ctype_of(t) for t in params]
        assert list(fn.argtypes) == want, f"{name}: binding {fn.argtypes} vs header {params}"
        assert fn.restype == _ctype_of(ret), f"{name}: binding returns {fn.restype}, header {ret}"
        checked += 1
    assert checked >= 19
