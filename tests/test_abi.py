"""The C ABI without a GPU: the library loads, exports every function that
include/moe.h declares, the ctypes mirrors match the C struct layouts, and the
host-side argument checks reject bad input before anything touches a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def moe(cuda_built):
    from routed_expert_decode_gb300 import moe as m

    m.lib()
    return m


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(moe):
    names = _declared_functions()
    assert "moe_layer" in names and "moe_route" in names and "moe_ffn" in names
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW]\s+(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(moe.lib(), n)


def test_struct_layouts_match_header(moe, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "moe.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(moe_mat), sizeof(moe_desc), sizeof(moe_weights),
         sizeof(moe_ws_layout));
  printf("%zu %zu %zu\n", offsetof(moe_desc, s), offsetof(moe_desc, flags),
         offsetof(moe_ws_layout, n_tap));
  printf("%zu %zu %zu\n", sizeof(moe_cache_stats), offsetof(moe_weights, expert_slot),
         offsetof(moe_weights, n_slots));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", HEADER_DIR, str(src), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sizes = [int(v) for v in lines[0].split()]
    offs = [int(v) for v in lines[1].split()]
    assert sizes == [ctypes.sizeof(moe.MoeMat), ctypes.sizeof(moe.MoeDesc),
                     ctypes.sizeof(moe.MoeWeights), ctypes.sizeof(moe.MoeWsLayout)]
    assert offs == [moe.MoeDesc.s.offset, moe.MoeDesc.flags.offset, moe.MoeWsLayout.n_tap.offset]
    cache = [int(v) for v in lines[2].split()]
    assert cache == [ctypes.sizeof(moe.MoeCacheStats), moe.MoeWeights.expert_slot.offset,
                     moe.MoeWeights.n_slots.offset]


def _desc(moe, **kw):
    base = dict(n_expert=256, top_k=8, d=6144, f=2048, f_shared=2048, routed_fmt=0, s=2.5)
    base.update(kw)
    return moe.make_desc(**base)


@pytest.mark.parametrize("bad", [dict(n_expert=0), dict(n_expert=1025), dict(top_k=0),
                                 dict(top_k=300), dict(n_expert=8, top_k=9), dict(d=100),
                                 dict(f=48), dict(f_shared=40), dict(routed_fmt=7),
                                 dict(top_k=33, n_expert=64), dict(s=float("nan"))])
def test_invalid_descriptors(moe, bad):
    d = _desc(moe, **bad)
    assert moe.lib().moe_workspace_size(ctypes.byref(d), 4) == 0
    lay = moe.MoeWsLayout()
    assert moe.lib().moe_workspace_layout(ctypes.byref(d), 4, ctypes.byref(lay)) == 1
    # rejected on the host before any launch (fake, never-dereferenced pointers)
    fake = ctypes.c_void_p(1 << 20)
    w = moe.MoeWeights()
    st = moe.lib().moe_layer(ctypes.byref(d), ctypes.byref(w), fake, fake, fake, 4, fake, fake,
                             1 << 30, None)
    assert st == 1
    st = moe.lib().moe_route(ctypes.byref(d), fake, fake, 4, fake, fake, fake, fake, fake,
                             None, 0, None)
    assert st == 1


def _weights(moe, align=256):
    w = moe.MoeWeights()
    base = 1 << 24
    for i, n in enumerate(("gate", "up", "down", "s_gate", "s_up", "s_down")):
        setattr(w, n, moe.MoeMat(base + i * (1 << 20) + align % 256, base + i * (1 << 20) + 64))
    return w


def test_host_checks_before_launch(moe):
    d = _desc(moe)
    lib = moe.lib()
    need = lib.moe_workspace_size(ctypes.byref(d), 4)
    assert need > 0
    fake = ctypes.c_void_p(1 << 22)
    good = _weights(moe)
    # workspace too small
    assert lib.moe_layer(ctypes.byref(d), ctypes.byref(good), fake, fake, fake, 4, fake, fake,
                         need - 1, None) == 3
    # misaligned weight codes (Q8_0 rows are read 32 bytes at a time)
    assert lib.moe_layer(ctypes.byref(d), ctypes.byref(_weights(moe, align=16)), fake, fake,
                         fake, 4, fake, fake, need, None) == 1
    # missing weights
    assert lib.moe_layer(ctypes.byref(d), ctypes.byref(moe.MoeWeights()), fake, fake, fake, 4,
                         fake, fake, need, None) == 1
    # misaligned workspace
    assert lib.moe_layer(ctypes.byref(d), ctypes.byref(good), fake, fake, fake, 4, fake,
                         ctypes.c_void_p((1 << 22) + 8), need, None) == 1
    # null inputs with T > 0
    assert lib.moe_layer(ctypes.byref(d), ctypes.byref(good), None, fake, fake, 4, fake, fake,
                         need, None) == 1
    assert lib.moe_ffn(ctypes.byref(d), ctypes.byref(good), fake, 4, None, fake, fake, fake,
                       fake, fake, fake, need, None) == 1
    # a NULL workspace names moe_layer_noalloc's static scratch: before any such
    # call nothing can have been flagged (and no CUDA call is made); a NULL
    # workspace with a size is a bad argument
    assert lib.moe_check_device_error(None, 0, None) == 0
    assert lib.moe_check_device_error(None, 4, None) == 1
    assert lib.moe_check_device_error(fake, 2, None) == 1


def test_workspace_layout_regions(moe):
    for T in (0, 1, 16, 512):
        for flags in (0, moe.FLAG_DEBUG_TAPS):
            d = _desc(moe, flags=flags)
            L = moe.workspace_layout(d, T)
            assert L.err == 0
            offs = [getattr(L, n) for n in moe.LAYOUT_FIELDS if n not in ("err", "total")
                    and (flags or not n.startswith("tap"))]
            assert all(o % 256 == 0 for o in offs)
            assert L.total == moe.workspace_size(d, T)
            assert L.total >= L.o + (T * 8 + T) * 6144 * 4
            assert L.n_tap == 8


def test_status_strings(moe):
    for st in range(7):
        assert moe.status_string(st)
    assert moe.status_string(99) == "unknown status"
