"""The C ABI library loads, exports every entry point include/*.h declares, and rejects
bad arguments on the host before touching a GPU (CPU only: no compute call is made)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from combine_moe_route_meta_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for n in ("moe_route_meta", "moe_dispatch", "moe_combine", "moe_status_string",
              "moe_route_meta_workspace_size", "moe_abi_version"):
        assert n in names, names


def test_diagnostics_live_in_their_own_header():
    """The hot-path boundary (moe_dispatch.h) declares no test hook; moe_diag.h holds them."""
    def declared(name):
        src = open(os.path.join(ROOT, "include", name)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        return set(re.findall(r"\b(moe_\w+)\s*\(", src))
    diag = {"moe_convert_probe", "moe_fp8_division_check", "moe_wait_timeout_check"}
    assert diag <= declared("moe_diag.h")
    assert not diag & declared("moe_dispatch.h")


def test_library_exports_every_declared_symbol(lib):
    from combine_moe_route_meta_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in _declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_package_imports_and_reports_version():
    import combine_moe_route_meta_gb300 as moe
    assert moe.moe_abi_version() == 1
    assert moe.moe_status_string(moe.MOE_ERR_CAPACITY).startswith("MOE_ERR_CAPACITY")
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_workspace_size_is_host_only():
    import combine_moe_route_meta_gb300 as moe
    assert moe.moe_route_meta_workspace_size(128, 8, 256) == 0          # one block
    n = moe.moe_route_meta_workspace_size(16384, 8, 128)                # 128 blocks x 128 experts
    assert n == 4 * 128 * 128                                           # int32 [B][E], nothing else
    assert moe.moe_route_meta_workspace_size(10, 17, 8) == 0            # K too large -> rejected
    assert moe.moe_route_meta_workspace_size(-1, 8, 8) == 0


def _c(lib, name):
    fn = getattr(lib, name)
    fn.restype = ctypes.c_int
    return fn


FAKE = ctypes.c_void_p(0x1000)       # never dereferenced: validation fails first


def test_route_meta_argument_validation(lib):
    f = _c(lib, "moe_route_meta")
    P = ctypes.c_void_p
    base = dict(ids=FAKE, T=4, K=2, E=8, P=1, M=0, seg=FAKE, s2d=FAKE, reo=FAKE, mm=FAKE)

    def call(**kw):
        a = dict(base, **kw)
        return f(a["ids"], ctypes.c_int64(a["T"]), a["K"], a["E"], a["P"], a["M"], a["seg"], a["s2d"],
                 a["reo"], a["mm"], None, None, None, ctypes.c_size_t(0), a.get("st", None), None)

    assert call(st=None) == 1                       # no status word
    assert call(K=0, st=FAKE) == 1
    assert call(K=17, st=FAKE) == 2                 # beyond MOE_MAX_TOPK
    assert call(E=2048, st=FAKE) == 2               # beyond MOE_MAX_EXPERTS
    assert call(E=8, P=3, st=FAKE) == 1             # E % P != 0
    assert call(M=-1, st=FAKE) == 1
    assert call(T=-1, st=FAKE) == 1
    assert call(seg=None, st=FAKE) == 1
    assert call(T=1 << 30, K=8, st=FAKE) == 2       # T*K beyond int32
    assert call(seg=ctypes.c_void_p(0x1004), st=FAKE) == 1   # misaligned int64 output
    # multi-block plan needs a workspace
    assert call(T=100000, st=FAKE) == 1


def test_dispatch_and_combine_argument_validation(lib):
    d = _c(lib, "moe_dispatch")
    d.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]

    def disp(mode=0, quant=0, x=FAKE, T=4, H=256, ids=FAKE, K=2, E=8, M=0, s2d=FAKE, seg=FAKE,
             q=FAKE, s=FAKE, st=FAKE):
        return d(mode, quant, x, T, H, ids, K, E, M, s2d, seg, 1.0, q, s, st, None)

    assert disp(mode=2) == 1
    assert disp(quant=7) == 1
    assert disp(quant=3, H=272) == 1                 # UE8M0 FP8 needs H % 128
    assert disp(H=100) == 1                          # H % 16
    assert disp(quant=1, H=272) == 1                 # fp8 needs H % 128
    assert disp(mode=1, M=0) == 1                    # masked needs M >= 1
    assert disp(st=None) == 1
    assert disp(x=ctypes.c_void_p(0x1008)) == 1      # 16-byte alignment of hidden_states
    assert disp(quant=1, s=None) == 1                # fp8 needs a scale buffer
    assert disp(mode=1, M=4, seg=None) == 1
    assert disp(T=0) == 0                            # empty batch: nothing to launch

    c = _c(lib, "moe_combine")
    c.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]

    def comb(mode=0, eo=FAKE, T=4, H=256, K=2, E=8, M=0, ids=FAKE, s2d=FAKE, seg=FAKE, w=FAKE, out=FAKE,
             st=FAKE):
        return c(mode, eo, T, H, K, E, M, ids, s2d, seg, w, out, st, None)

    assert comb(H=8) == 1
    assert comb(w=None) == 1
    assert comb(out=ctypes.c_void_p(0x1002)) == 1
    assert comb(mode=1, M=0) == 1
    assert comb(K=20) == 2
    assert comb(T=0) == 0


def test_swizzled_scale_layout_validation(lib):
    """MOE_SCALES_SWIZZLED_128X4: NVFP4 only, H % 64 == 0, 4-byte aligned scales."""
    d = _c(lib, "moe_dispatch_ex")
    d.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]

    def disp(layout=2, quant=2, T=4, H=256, s=FAKE):
        return d(0, quant, layout, FAKE, T, H, FAKE, 2, 8, 0, 0, FAKE, FAKE, 1.0, FAKE, s, FAKE, None)

    assert disp(quant=1) == 1                      # FP8 has no swizzled layout
    assert disp(H=272) == 1                        # 17 scale columns: not whole 4-column tiles
    assert disp(s=ctypes.c_void_p(0x1002)) == 1    # scales must be 4-byte aligned
    assert disp(layout=3) == 1
    assert disp(T=0) == 0
    p = _c(lib, "moe_dispatch_partitioned_ex")
    p.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int32,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]

    def part(quant=2, layout=2, H=256, S=0, sf=FAKE):
        return p(quant, layout, FAKE, 0, S, H, FAKE, FAKE, 2, 8, 2, -1, 1.0, FAKE, sf, FAKE, FAKE, FAKE, None)

    assert part(quant=0) == 1                      # bf16 payload has no scales to swizzle
    assert part(layout=1) == 1                     # column-major is an FP8 layout
    assert part(H=80) == 1
    assert part(sf=ctypes.c_void_p(0x1001)) == 1
    assert part() == 0                             # no slots: nothing to launch


def test_division_check_validation(lib):
    f = _c(lib, "moe_fp8_division_check")
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert f(None, None) == 1
    assert f(ctypes.c_void_p(0x1004), None) == 1      # 8-byte alignment


def test_wait_timeout_check_validation(lib):
    f = _c(lib, "moe_wait_timeout_check")
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    st = ctypes.c_void_p(0x1000)
    assert f(None, 1000, 0, None) == 1                 # no status word
    assert f(ctypes.c_void_p(0x1002), 1000, 0, None) == 1  # 4-byte alignment
    assert f(st, 0, 0, None) == 1                      # limit in 1 .. 10^10 ns
    assert f(st, 10 ** 10 + 1, 0, None) == 1
    assert f(st, 1000, 2, None) == 1                   # complete is 0 or 1
