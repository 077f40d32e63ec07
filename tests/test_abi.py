"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and its host-only functions size, lay out and reject inputs
without launching anything."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

import expert_routing_alignment_gb300 as moe
import oracle
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(moe_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_align", "moe_grouped_gate_up", "moe_grouped_down", "moe_blend",
                     "moe_decode_layer", "moe_topk_softmax", "moe_align_sizes",
                     "moe_decode_layer_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = moe.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(moe.EXPORTS)


def test_version_and_status_strings():
    lib = moe.load()
    assert b"sm_103a" in lib.moe_version()
    assert lib.moe_status_string(moe.MOE_EINVAL) == b"invalid argument"


@pytest.mark.parametrize("n,E,BS", [(0, 8, 16), (1, 64, 16), (64, 128, 16), (1024, 256, 64),
                                    (32768, 1024, 128), (8, 4, 1)])
def test_align_sizes_match_oracle(n, E, BS):
    assert moe.moe_align_sizes(n, E, BS) == oracle.align_sizes(n, E, BS)


def test_align_sizes_rejects():
    lib = moe.load()
    a = ctypes.c_int()
    for args in [(-1, 8, 16), (8, 0, 16), (8, 8, 0)]:
        assert lib.moe_align_sizes(*args, ctypes.byref(a), ctypes.byref(a),
                                   ctypes.byref(a)) == moe.MOE_EINVAL
    assert lib.moe_align_sizes((1 << 20) + 1, 8, 16, ctypes.byref(a), ctypes.byref(a),
                               ctypes.byref(a)) == moe.MOE_EUNSUPPORTED
    assert lib.moe_align_sizes(8, 8, 16, None, None, None) == moe.MOE_EINVAL


def test_align_rejects_before_launch():
    lib = moe.load()
    fake = ctypes.c_void_p(256)
    # NULL tables, too many experts: rejected on the host (nothing launched)
    args = [fake, 0, 8, 8, 16] + [fake] * 4 + [None] + [fake] * 3 + [None]
    assert lib.moe_align(*args) == moe.MOE_EINVAL
    args = [fake, 0, 8, 2048, 16] + [fake] * 8 + [None]
    assert lib.moe_align(*args) == moe.MOE_EUNSUPPORTED


class _FakeTensor:
    """Stands in for a device tensor: only its address is read on the host."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _fake_experts(fmt=moe.FMT_FP8_B128, E=128, H=2048, I=768, align=256):
    t = lambda: _FakeTensor(align)
    g = None if fmt == moe.FMT_FP8_B128 else _FakeTensor(align)
    proj = (t(), t(), g)
    return moe.Experts(fmt, E, H, I, proj, proj, proj)


def test_workspace_layout_host_only():
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts())
    nb = moe.workspace_bytes(layer, 8)
    v = moe._WsView()
    lib = moe.load()
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), 8,
                                               ctypes.byref(v)) == 0
    assert v.total_bytes == nb
    mt, mb, cap = oracle.align_sizes(64, 128, 16)
    assert (v.max_total, v.max_blocks, v.cap) == (mt, mb, cap)
    offs = [v.topk_ids, v.topk_w, v.sorted_token_ids, v.sorted_expert_ids, v.expert_offsets,
            v.token_to_perm, v.active_experts, v.active_count, v.num_tokens_post_padded, v.h,
            v.h_shared, v.y, v.y_shared]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert v.y - v.h >= mt * 768 * 4 and nb - v.y >= mt * 2048 * 4
    # workspace grows with M
    assert moe.workspace_bytes(layer, 1) < nb < moe.workspace_bytes(layer, 128)


def test_tensor_core_workspace_host_only():
    """FP8 routed experts without a shared expert get the tensor-core term
    tables appended to the workspace: [2][max_total][H] and [3][max_total][I]
    E4M3 planes, their float scales and a per-active-expert count."""
    lib = moe.load()
    layer = moe.LayerDesc(top_k=8, block_size=64, routed=_fake_experts(E=256, H=4096, I=1536))
    v = moe._WsView()
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), 128,
                                               ctypes.byref(v)) == 0
    mt, _, cap = oracle.align_sizes(1024, 256, 64)
    offs = [v.blend_counters, v.tc_done, v.tc_x_terms, v.tc_x_scale, v.tc_h_terms, v.tc_h_scale]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    # the counters that persist between calls come first: [0, 8) and 256.. (E + 1 ints)
    assert v.blend_counters == 0 and v.tc_done == 256
    assert v.topk_ids - v.tc_done >= (256 + 1) * 4
    assert v.tc_x_scale - v.tc_x_terms >= 2 * mt * 4096
    assert v.tc_h_terms - v.tc_x_scale >= mt * 4
    assert v.tc_h_scale - v.tc_h_terms >= 3 * mt * 1536
    assert v.total_bytes - v.tc_h_scale >= mt * 12 * 4
    assert moe.workspace_bytes(layer, 128) == v.total_bytes
    # ... at offsets that do not move with M, so one workspace serves every M
    for M in (1, 8, 64):
        w = moe._WsView()
        assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), M,
                                                   ctypes.byref(w)) == 0
        assert (w.blend_counters, w.tc_done) == (0, 256)
    # the tensor-core run is 3 launches with router logits, 2 with given ids
    assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), 128, 1) == 3
    assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), 128, 0) == 2
    # not when the CUDA-core path is forced
    lay = moe.LayerDesc(top_k=8, block_size=64, path=moe.PATH_SIMT_STAGED,
                        routed=_fake_experts(E=256, H=4096, I=1536))
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(lay._struct), 128,
                                               ctypes.byref(v)) == 0
    assert v.tc_x_terms == v.tc_h_terms == v.tc_done == 0
    # NVFP4 experts at M = 128 run on the CUDA cores: no term tables, but the
    # counters of the NVFP4 tensor-core kernel (M <= 32) keep their place
    lay = moe.LayerDesc(top_k=8, block_size=64,
                        routed=_fake_experts(fmt=moe.FMT_NVFP4_G16, E=256, H=4096, I=1536))
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(lay._struct), 128,
                                               ctypes.byref(v)) == 0
    assert v.tc_x_terms == v.tc_h_terms == v.tc_items == 0 and v.tc_done == 256


def test_nvfp4_tensor_core_workspace_host_only():
    """NVFP4 routed experts at M <= 32 get the NVFP4 tensor-core kernel's
    tables: an f16 x table of 16 or 32 token columns, [2][max_total][I] f16
    h terms (then the FP8 shared expert's [2][32][Is]), their scales and
    the active table; the counters (E + 2 ints) at 256 for every M.  The
    shared expert runs in the same kernel: the launch count does not
    change with it."""
    lib = moe.load()
    shared = _fake_experts(E=1, H=2048, I=512)
    for sh in (None, shared):
        layer = moe.LayerDesc(top_k=8, block_size=16, shared=sh,
                              routed=_fake_experts(fmt=moe.FMT_NVFP4_G16, E=128, H=2048, I=768))
        for M in (1, 8, 16, 17, 32, 33, 64):
            v = moe._WsView()
            assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), M,
                                                       ctypes.byref(v)) == 0
            mt, _, cap = oracle.align_sizes(M * 8, 128, 16)
            assert (v.blend_counters, v.tc_done) == (0, 256)
            assert v.topk_ids - v.tc_done >= (128 + 2) * 4
            launches = lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), M, 1)
            if M > 32:   # the CUDA cores
                assert v.tc_x_terms == v.tc_h_terms == v.tc_items == 0
                continue
            assert v.tc_x_scale - v.tc_x_terms >= 2 * 32 * 2048
            assert v.tc_h_terms - v.tc_x_scale >= 32 * 4
            Is = 512 if sh is not None else 0
            assert v.tc_h_scale - v.tc_h_terms >= 2 * 2 * (mt * 768 + 32 * Is)
            assert v.tc_items - v.tc_h_scale >= (mt * 6 + 32 * (Is // 128)) * 4
            assert v.total_bytes - v.tc_items >= cap * 16
            assert launches == 3
            assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), M, 0) == 2


def test_token_form_workspace_host_only():
    """FP8 batches of M <= 16 on the tensor-core path keep their x terms by
    token: a [H/128][2][16][128] table and 16 scales, whatever max_total is;
    above 16 rows they are by sorted row.  The counters sit at 256 either way."""
    lib = moe.load()
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts(E=128, H=2048, I=768))
    for M in (1, 8, 16, 17):
        v = moe._WsView()
        assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), M,
                                                   ctypes.byref(v)) == 0
        mt, _, cap = oracle.align_sizes(M * 8, 128, 16)
        rows = 16 if M <= 16 else mt
        assert (v.blend_counters, v.tc_done) == (0, 256)
        assert v.tc_x_scale - v.tc_x_terms >= 2 * rows * 2048
        assert v.tc_h_terms - v.tc_x_scale >= rows * 4
        assert v.total_bytes - v.tc_items >= cap * 16
        assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), M, 1) == 3


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=moe.FMT_FP8_B128, H=2000), moe.MOE_EUNSUPPORTED),   # FP8 needs H % 128
    (dict(fmt=moe.FMT_NVFP4_G16, I=784), moe.MOE_EUNSUPPORTED),   # NVFP4 needs I % 32
    (dict(fmt=7), moe.MOE_EINVAL),
    (dict(E=1025), moe.MOE_EUNSUPPORTED),
    (dict(align=8), moe.MOE_EINVAL),                              # codes not 16-byte aligned
])
def test_layer_shape_admission(kw, status):
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts(**kw))
    v = moe._WsView()
    got = moe.load().moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), 8,
                                                     ctypes.byref(v))
    assert got == status


def test_layer_rejects_rows_and_topk():
    lib = moe.load()
    v = moe._WsView()
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts())
    p = ctypes.pointer(layer._struct)
    assert lib.moe_decode_layer_workspace_view(p, 0, ctypes.byref(v)) == moe.MOE_EINVAL
    # above 128 rows only on the tensor-core path, up to 4096
    assert lib.moe_decode_layer_workspace_view(p, 129, ctypes.byref(v)) == 0
    assert lib.moe_decode_layer_workspace_view(p, 4096, ctypes.byref(v)) == 0
    assert lib.moe_decode_layer_workspace_view(p, 4097, ctypes.byref(v)) == moe.MOE_EUNSUPPORTED
    simt = moe.LayerDesc(top_k=8, block_size=16, path=moe.PATH_SIMT, routed=_fake_experts())
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(simt._struct), 129,
                                               ctypes.byref(v)) == moe.MOE_EUNSUPPORTED
    nv = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts(fmt=moe.FMT_NVFP4_G16))
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(nv._struct), 129,
                                               ctypes.byref(v)) == moe.MOE_EUNSUPPORTED
    bad_k = moe.LayerDesc(top_k=200, block_size=16, routed=_fake_experts())
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(bad_k._struct), 8,
                                               ctypes.byref(v)) == moe.MOE_EINVAL
    # moe_decode_layer itself rejects a short workspace before any launch
    fake = ctypes.c_void_p(256)
    assert lib.moe_decode_layer(p, fake, 8, fake, None, None, fake, fake, 16, None,
                                None) == moe.MOE_EINVAL


def test_hidden_in_launch_counts_and_logits_region():
    """A layer with router weights can take x alone: the logits kernel runs
    ahead of the route (one launch more than with given logits) and writes
    the [M][E] float router_logits region of the workspace."""
    lib = moe.load()
    fake_w = torch.zeros(16, dtype=torch.int64)   # a host address; nothing is launched
    for path, with_l in ((moe.PATH_AUTO, 3), (moe.PATH_SIMT_STAGED, 5)):
        plain = moe.LayerDesc(top_k=8, block_size=64, path=path,
                              routed=_fake_experts(E=256, H=4096, I=1536))
        assert lib.moe_decode_layer_launches(ctypes.pointer(plain._struct), 128, 2) == -1
        layer = moe.LayerDesc(top_k=8, block_size=64, path=path, router_weight=fake_w,
                              routed=_fake_experts(E=256, H=4096, I=1536))
        assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), 128, 1) == with_l
        assert lib.moe_decode_layer_launches(ctypes.pointer(layer._struct), 128, 2) == with_l + 1
        v = moe._WsView()
        assert lib.moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), 128,
                                                   ctypes.byref(v)) == 0
        assert v.router_logits % 256 == 0 and v.router_logits > v.blend_counters
        nxt = [o for o in (v.tc_x_terms, v.total_bytes) if o > v.router_logits]
        assert min(nxt) - v.router_logits >= 128 * 256 * 4


def test_shared_gate_needs_a_shared_expert():
    lib = moe.load()
    gate = torch.zeros(2048, dtype=torch.int16)   # a host address; nothing is launched
    lay = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts(E=128, H=2048, I=768),
                        shared_gate=gate)
    v = moe._WsView()
    assert lib.moe_decode_layer_workspace_view(ctypes.pointer(lay._struct), 8,
                                               ctypes.byref(v)) == moe.MOE_EINVAL


def test_header_is_plain_c_and_struct_layouts_match_the_binding(tmp_path):
    """The header compiles as C99, and the binding's ctypes mirrors have the
    header's sizes and field offsets (a C program prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    structs = {"moe_layer_desc": moe._LayerDesc, "moe_workspace_view": moe._WsView,
               "moe_experts": moe._Experts, "moe_proj": moe._Proj}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe_gb300.h"',
             "int main(void) {"]
    for cname, cty in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cty._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {tuple(l.split()[:-1]): int(l.split()[-1]) for l in out.splitlines()}
    for cname, cty in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cty), cname
        for fname, _ in cty._fields_:
            assert got[(cname, fname)] == getattr(cty, fname).offset, (cname, fname)


def test_a_c_program_links_the_library_and_gets_the_bindings_answers(tmp_path):
    """The library is usable from plain C: a C99 program includes the header,
    links the shared library and calls the host-only entry points; its
    answers equal the Python binding's (and the oracle's sizes)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = moe.load()._name
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include "moe_gb300.h"
static unsigned char codes[256] __attribute__((aligned(256)));
static float scales[64] __attribute__((aligned(256)));
int main(void) {
    int mt = 0, mb = 0, cap = 0;
    if (moe_align_sizes(64, 128, 16, &mt, &mb, &cap) != MOE_OK) return 2;
    printf("sizes %d %d %d\n", mt, mb, cap);
    printf("einval %s\n", moe_status_string(MOE_EINVAL));
    moe_layer_desc L = {0};
    L.top_k = 8;
    L.block_size = 16;
    L.path = MOE_PATH_AUTO;
    L.routed.fmt = MOE_FMT_FP8_B128;
    L.routed.num_experts = 128;
    L.routed.hidden = 2048;
    L.routed.inter = 768;
    moe_proj p = {codes, scales, NULL};
    L.routed.gate = p;
    L.routed.up = p;
    L.routed.down = p;
    printf("ws %zu\n", moe_decode_layer_workspace_bytes(&L, 8));
    printf("launches %d %d\n", moe_decode_layer_launches(&L, 8, 1),
           moe_decode_layer_launches(&L, 8, 0));
    return 0;
}
''')
    exe = tmp_path / "use"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    str(src), so, "-Wl,-rpath," + os.path.dirname(so), "-o", str(exe)],
                   check=True, capture_output=True)
    out = dict(l.split(" ", 1) for l in
               subprocess.run([str(exe)], check=True, capture_output=True,
                              text=True).stdout.splitlines())
    assert tuple(map(int, out["sizes"].split())) == tuple(oracle.align_sizes(64, 128, 16))
    assert out["einval"] == moe.load().moe_status_string(moe.MOE_EINVAL).decode()
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts())
    assert int(out["ws"]) == moe.workspace_bytes(layer, 8)
    assert out["launches"].split() == [str(moe.moe_decode_layer_launches(layer, 8, 1)),
                                       str(moe.moe_decode_layer_launches(layer, 8, 0))]


def test_router_blend_and_noalloc_reject_before_launch():
    """Host checks of the router, the gated blend and the no-alloc layer:
    each rejection returns before anything is launched (fake addresses)."""
    lib = moe.load()
    f = ctypes.c_void_p(4096)        # 16-byte aligned
    odd = ctypes.c_void_p(4096 + 8)  # 8-byte aligned only
    # router: NULL / sizes, hidden % 8, misaligned operands
    assert lib.moe_router_logits(None, f, 2, 256, 8, f, None) == moe.MOE_EINVAL
    assert lib.moe_router_logits(f, f, 0, 256, 8, f, None) == moe.MOE_EINVAL
    assert lib.moe_router_logits(f, f, 2, 100, 8, f, None) == moe.MOE_EUNSUPPORTED
    assert lib.moe_router_logits(odd, f, 2, 256, 8, f, None) == moe.MOE_EUNSUPPORTED
    assert lib.moe_router_logits(f, odd, 2, 256, 8, f, None) == moe.MOE_EUNSUPPORTED
    # blend: a gate needs the shared term and x; gated needs hidden % 8 and alignment
    assert lib.moe_blend(f, f, f, None, f, f, f, 2, 1, 256, None) == moe.MOE_EINVAL
    assert lib.moe_blend(f, f, f, f, None, f, f, 2, 1, 256, None) == moe.MOE_EINVAL
    assert lib.moe_blend(f, f, f, f, f, f, f, 2, 1, 260, None) == moe.MOE_EUNSUPPORTED
    assert lib.moe_blend(f, f, f, f, f, odd, f, 2, 1, 256, None) == moe.MOE_EUNSUPPORTED
    # no-alloc layer: a workspace above the fixed array is rejected (verify batch)
    layer = moe.LayerDesc(top_k=8, block_size=64, routed=_fake_experts(E=256, H=4096, I=1536))
    assert moe.workspace_bytes(layer, 128) > moe.NOALLOC_SCRATCH_BYTES
    assert lib.moe_decode_layer_noalloc(ctypes.pointer(layer._struct), f, 128, f, None, None,
                                        f, None, None) == moe.MOE_EUNSUPPORTED
    # the layer: hidden in with misaligned router weights
    bad = moe.LayerDesc(top_k=8, block_size=16, routed=_fake_experts(),
                        router_weight=_FakeTensor(4096 + 8))
    ws = ctypes.c_void_p(1 << 20)
    assert lib.moe_decode_layer(ctypes.pointer(bad._struct), f, 8, None, None, None, f, ws,
                                moe.workspace_bytes(bad, 8), None, None) == moe.MOE_EINVAL


def test_binding_refuses_buffers_the_c_abi_cannot_read():
    """The Python wrappers refuse wrong dtypes, shapes and strided views before
    any call into the library."""
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    w = torch.zeros(8, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        moe.moe_router_logits(x.float(), w)
    with pytest.raises(ValueError):
        moe.moe_router_logits(x, w[:, :128])
    with pytest.raises(ValueError):
        moe.moe_router_logits(torch.zeros(4, 512, dtype=torch.bfloat16)[:, ::2], w)
    with pytest.raises(ValueError):
        moe.moe_router_logits(x, w, torch.zeros(4, 8, dtype=torch.float64))
    y = torch.zeros(8, 256)
    out = torch.zeros(4, 256, dtype=torch.bfloat16)
    ttp = torch.zeros(4, dtype=torch.int32)
    tw = torch.ones(4, 1)
    with pytest.raises(ValueError):
        moe.moe_blend(y, tw, ttp, y[:4], out, 1, x=None, shared_gate=torch.zeros(256))
    with pytest.raises(ValueError):
        moe.moe_blend(y, tw, ttp, y[:4], out, 1, x=x,
                      shared_gate=torch.zeros(256, dtype=torch.float32))
    with pytest.raises(ValueError):
        moe.moe_blend(y, tw, ttp, y[:4], out, 1, x=x,
                      shared_gate=torch.zeros(128, dtype=torch.bfloat16))


def _header_params(fn: str) -> list:
    """Parameter names of fn's declaration in the header, in order."""
    text = open(os.path.join(ROOT, "include", "moe_gb300.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    m = re.search(r"\b" + fn + r"\s*\(([^;]*?)\)\s*;", text, flags=re.S)
    assert m, fn
    return [re.findall(r"\w+", p)[-1] for p in m.group(1).split(",")]


class _Recorder:
    """Stands in for the library: records each call's arguments."""

    def __init__(self):
        self.calls = {}

    def __getattr__(self, name):
        def call(*args):
            self.calls[name] = args
            return 0
        return call


def _val(a):
    return a.value if isinstance(a, ctypes.c_void_p) else a


@pytest.mark.parametrize("fn", ["moe_router_logits", "moe_blend", "moe_topk_softmax",
                                "moe_decode_layer", "moe_decode_layer_noalloc", "moe_align",
                                "moe_grouped_gate_up", "moe_grouped_down",
                                "moe_decode_experts"])
def test_binding_passes_arguments_in_the_headers_order(monkeypatch, fn):
    rec = _Recorder()
    monkeypatch.setattr(moe, "_lib", rec)
    M, H, E, k = 4, 256, 8, 2
    x = torch.zeros(M, H, dtype=torch.bfloat16)
    if fn == "moe_router_logits":
        W = torch.zeros(E, H, dtype=torch.bfloat16)
        lg = torch.zeros(M, E)
        moe.moe_router_logits(x, W, lg, stream=7)
        want = dict(x=x, router_weight=W, M=M, hidden=H, num_experts=E, logits=lg)
    elif fn == "moe_blend":
        y, w, ttp = torch.zeros(16, H), torch.zeros(M, k), torch.zeros(M * k, dtype=torch.int32)
        ysh, g = torch.zeros(M, H), torch.zeros(H, dtype=torch.bfloat16)
        out = torch.zeros(M, H, dtype=torch.bfloat16)
        moe.moe_blend(y, w, ttp, ysh, out, k, x=x, shared_gate=g, stream=7)
        want = dict(y=y, topk_w=w, token_to_perm=ttp, y_shared=ysh, x=x, shared_gate=g,
                    out=out, M=M, top_k=k, hidden=H)
    elif fn == "moe_topk_softmax":
        lg = torch.zeros(M, E)
        ids, w = moe.moe_topk_softmax(lg, k, stream=7)
        want = dict(logits=lg, M=M, num_experts=E, top_k=k, topk_ids=ids, topk_w=w)
    elif fn == "moe_decode_layer":
        layer = moe.LayerDesc(top_k=k, block_size=16, routed=_fake_experts(E=E, H=H, I=256))
        out = torch.zeros(M, H, dtype=torch.bfloat16)
        ws = torch.zeros(1024, dtype=torch.uint8)
        lg, err = torch.zeros(M, E), torch.zeros(1, dtype=torch.int32)
        moe.moe_decode_layer(layer, x, out, ws, router_logits=lg, err_word=err, stream=7)
        want = dict(x=x, M=M, router_logits=lg, topk_ids=None, topk_w=None, out=out,
                    workspace=ws, workspace_bytes=1024, err_word=err)
    elif fn == "moe_decode_experts":
        layer = moe.LayerDesc(top_k=k, block_size=16, routed=_fake_experts(E=E, H=H, I=256))
        out = torch.zeros(M, H, dtype=torch.bfloat16)
        ws = torch.zeros(1024, dtype=torch.uint8)
        err = torch.zeros(1, dtype=torch.int32)
        moe.moe_decode_experts(layer, x, out, ws, err_word=err, stream=7)
        want = dict(x=x, M=M, out=out, workspace=ws, workspace_bytes=1024, err_word=err)
    elif fn == "moe_decode_layer_noalloc":
        layer = moe.LayerDesc(top_k=k, block_size=16, routed=_fake_experts(E=E, H=H, I=256))
        out = torch.zeros(M, H, dtype=torch.bfloat16)
        ids, w = torch.zeros(M, k, dtype=torch.int32), torch.zeros(M, k)
        err = torch.zeros(1, dtype=torch.int32)
        moe.moe_decode_layer_noalloc(layer, x, out, topk_ids=ids, topk_w=w, err_word=err,
                                     stream=7)
        want = dict(x=x, M=M, router_logits=None, topk_ids=ids, topk_w=w, out=out, err_word=err)
    elif fn == "moe_align":
        ids = torch.zeros(M * k, dtype=torch.int64)
        err = torch.zeros(1, dtype=torch.int32)
        t = moe.moe_align(ids, E, 16, err_word=err, stream=7)
        want = dict(topk_ids=ids, ids_is_int64=1, n=M * k, num_experts=E, block_size=16,
                    err_word=err, **{key: t[key] for key in (
                        "sorted_token_ids", "sorted_expert_ids", "expert_offsets",
                        "token_to_perm", "active_experts", "active_count",
                        "num_tokens_post_padded")})
    else:
        routed = _fake_experts(E=E, H=H, I=256)
        mt, _, cap = oracle.align_sizes(M * k, E, 16)
        i32 = dict(dtype=torch.int32)
        t = dict(expert_offsets=torch.zeros(E + 1, **i32), sorted_token_ids=torch.zeros(mt, **i32),
                 active_experts=torch.zeros(cap, **i32), active_count=torch.zeros(1, **i32))
        tabs = dict(t)
        h, y = torch.zeros(mt, 256), torch.zeros(mt, H)
        if fn == "moe_grouped_gate_up":
            moe.moe_grouped_gate_up(routed, None, x, k, t, h, None, path=moe.PATH_SIMT, stream=7)
            want = dict(x=x, M=M, top_k=k, h=h, h_shared=None, path=moe.PATH_SIMT, **tabs)
        else:
            moe.moe_grouped_down(routed, None, h, None, M, k, t, y, None, path=moe.PATH_SIMT,
                                 stream=7)
            want = dict(h=h, h_shared=None, M=M, top_k=k, y=y, y_shared=None,
                        path=moe.PATH_SIMT, **tabs)
    names = _header_params(fn)
    got = dict(zip(names, rec.calls[fn]))
    assert len(rec.calls[fn]) == len(names)
    assert _val(got["stream"]) == 7
    for name, v in want.items():
        exp = v.data_ptr() if isinstance(v, torch.Tensor) else v
        assert _val(got[name]) == exp, name
