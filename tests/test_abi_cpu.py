"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe_gb300.h declares, and rejects bad arguments
before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_moe_expert_gb300 import _build
    _build.build()
    import sparse_moe_expert_gb300 as moe
    return moe.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**\s*(moe_[a-z0-9_]+)\s*\(",
                                    src, re.M))
    return names


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert len(names) >= 11, names
    import sparse_moe_expert_gb300 as moe
    assert names == set(moe.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    import sparse_moe_expert_gb300 as moe
    assert moe.moe_abi_version() == 2
    assert moe.moe_status_string(0) == "ok"
    assert moe.moe_status_string(3) == "gate and up cannot be fused"
    assert moe.moe_status_string(99) == "unknown status"


def vp(v):
    return ctypes.c_void_p(v)


GOOD = 0x10000  # an aligned fake address; never dereferenced by a rejected call


def test_router_rejects_bad_shapes_before_launch(L):
    f = L.moe_router_topk
    args = dict(x=GOOD, w=GOOD, b=None, it=1.0, T=4, H=256, E=8, k=2, kmax=2, t1=1.2, t2=2.5, rn=1,
                ids=GOOD, tw=GOOD, kd=GOOD, me=GOOD, ws=GOOD, wsb=1 << 20)

    def call(**over):
        a = dict(args, **over)
        return f(vp(a["x"]), vp(a["w"]), a["b"], ctypes.c_float(a["it"]), a["T"], a["H"], a["E"],
                 a["k"], a["kmax"], ctypes.c_float(a["t1"]), ctypes.c_float(a["t2"]), a["rn"],
                 vp(a["ids"]), vp(a["tw"]), vp(a["kd"]), vp(a["me"]), vp(a["ws"]), a["wsb"], None)
    assert call(H=100) == 1          # H % 64
    assert call(E=0) == 1
    assert call(E=2000) == 1
    assert call(k=3) == 1            # k > kmax
    assert call(k=0, kmax=2) == 1    # adaptive needs kmax >= 3
    assert call(kmax=17) == 1
    assert call(x=GOOD + 4) == 1     # misaligned
    assert call(wsb=0) == 1          # workspace too small
    assert call(t1=3.0, t2=2.0) == 1
    assert call(kd=0) == 1


def test_qmm_and_pack_reject_before_launch(L):
    import sparse_moe_expert_gb300 as moe
    g = L.moe_gate_up_qmm
    base = [vp(GOOD), vp(GOOD), vp(GOOD), vp(GOOD), 4, 2, 8, 256, 512, vp(GOOD), vp(GOOD),
            vp(GOOD)]
    assert g(*base, 3, 1, 0, vp(GOOD), 0, None) == 2                    # bits 3 unsupported
    gated = moe.PATH_GEMV | moe.path_k_range(1, 2)
    for bits in (5, 6):           # the GEMV family only, and without a k gate
        assert g(*base, bits, 1, 0, vp(GOOD), moe.PATH_TC, None) == 2
        assert g(*base, bits, 1, 0, vp(GOOD), gated, None) == 2
    assert g(*base, 4, 0, 1, vp(GOOD), 0, None) == 2                    # RAW needs fp32 out
    assert g(*base, 4, 7, 0, vp(GOOD), 0, None) == 1                    # bad epilogue
    assert g(*base, 4, 1, 0, vp(GOOD), 9, None) == 1                    # bad path
    bad = list(base)
    bad[7] = 200                                                        # H % 64
    assert g(*bad, 4, 1, 0, vp(GOOD), 0, None) == 1
    d = L.moe_down_qmm
    assert d(vp(GOOD), 0, vp(GOOD), vp(GOOD), 4, 2, 8, 100, 256, vp(GOOD), vp(GOOD), vp(GOOD), 4,
             vp(GOOD), 0, 0, None) == 1                                 # I % 64
    assert d(vp(GOOD), 0, vp(GOOD), vp(GOOD), 4, 2, 8, 128, 256, vp(GOOD), vp(GOOD), vp(GOOD), 4,
             vp(GOOD), 5, 0, None) == 1                                 # bad y dtype
    a = moe.qdesc(512, 256, 4)
    for field, val in [("bits", 8), ("group_size", 32), ("has_bias", 1), ("rows", 256),
                       ("cols", 512), ("mode", 1), ("quantized", 0), ("scale_dtype", 1)]:
        b = moe.qdesc(512, 256, 4)
        setattr(b, field, val)
        st = L.moe_pack_gate_up(ctypes.byref(a), ctypes.byref(b), *[vp(GOOD)] * 6, 8,
                                *[vp(GOOD)] * 3, None)
        assert st == 3, field                                           # MOE_ERR_INCOMPATIBLE
    c = moe.qdesc(512, 256, 3)
    st = L.moe_pack_gate_up(ctypes.byref(c), ctypes.byref(c), *[vp(GOOD)] * 6, 8, *[vp(GOOD)] * 3,
                            None)
    assert st == 2                                                      # bits 3 unsupported
    assert L.moe_permute(vp(GOOD), vp(GOOD), 4, 2, 0, vp(GOOD), vp(GOOD), vp(GOOD), vp(GOOD),
                         None) == 1
    assert L.moe_combine(vp(GOOD), 0, vp(GOOD), vp(GOOD), vp(GOOD), 4, 2, 100, vp(GOOD),
                         None) == 1                                     # H % 64
    assert L.moe_combine(vp(GOOD), 7, vp(GOOD), vp(GOOD), vp(GOOD), 4, 2, 128, vp(GOOD),
                         None) == 1                                     # bad y dtype
    assert L.moe_swiglu(vp(GOOD), vp(GOOD), vp(GOOD), 4, 2, 256, 5, vp(GOOD), None) == 1


def test_workspace_size_grows_with_tokens(L):
    import sparse_moe_expert_gb300 as moe
    assert moe.moe_router_workspace_size(0) > 0
    assert moe.moe_router_workspace_size(4096) >= 2 * 4 * 4096


def test_header_constants_match_the_binding(tmp_path):
    """The header compiles as C, and its path flags, k-range macro, dropped
    marker and dtype codes agree with the Python binding's constants."""
    import shutil
    import subprocess
    import sparse_moe_expert_gb300 as moe
    from sparse_moe_expert_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consts.c"
    src.write_text(
        '#include <stdio.h>\n#include "moe_gb300.h"\n'
        "int main(void) {\n"
        '  printf("%d %d %d %d %d %d %d\\n", MOE_PATH_GEMV, MOE_PATH_TC, MOE_PATH_FLAG_WEIGHTS_EARLY,\n'
        "         MOE_PATH_FLAG_K_GATED, MOE_PATH_K_RANGE(2, 3), MOE_DROPPED, MOE_PATH_AUTO);\n"
        "  return 0;\n}\n")
    exe = tmp_path / "consts"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals == [moe.PATH_GEMV, moe.PATH_TC, moe.PATH_FLAG_WEIGHTS_EARLY,
                    moe.PATH_FLAG_K_GATED, moe.path_k_range(2, 3), moe.DROPPED,
                    moe.PATH_AUTO]
