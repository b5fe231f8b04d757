"""Host-side checks of the C ABI (no GPU needed, no kernel launched): the
library loads, exports every function its headers declare, sizes the
workspace, selects kernels deterministically, and rejects bad arguments
with a status before touching the device."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from sparse_mask_transformer_gb300 import build as stof_build
from sparse_mask_transformer_gb300 import stof

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    stof_build.build()
    return stof.load_library()


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(stof_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared("stof.h")
    assert set(stof.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    synth = ctypes.CDLL(stof.SYNTH_LIB_PATH)
    for n in _declared("stof_synth.h"):
        assert hasattr(synth, n), n


def test_version_and_status_strings(lib):
    assert stof.stof_version() == 3
    for s in range(10):
        assert stof.stof_status_string(s)
    assert "unknown" in stof.stof_status_string(99)


def test_struct_layout_matches_header(lib):
    # int32 x 8, 7 pointers, int64 x 4
    assert ctypes.sizeof(stof.stof_format) == 8 * 4 + 7 * 8 + 4 * 8


def test_workspace_bytes(lib):
    ws = stof.stof_encode_workspace_bytes
    # 16384^2 x 32 masks at 128x128: 524288 tiles x (2 KB bitmap + 8 B indices + 1 class byte)
    # + row pointers and per-row counts
    n = ws(32, 16384, 16384, 128, 128)
    tiles = 32 * 128 * 128
    assert tiles * (2048 + 8 + 1) <= n <= tiles * (2048 + 8 + 1) + (1 << 20)
    assert ws(1, 256, 256, 16, 16) > 0
    assert ws(1, 250, 256, 16, 16) == ws(1, 256, 256, 16, 16)  # a side not a whole number of OTs is padded
    assert ws(1, 256, 256, 12, 16) == 0      # bm not a multiple of 8
    assert ws(1, 512, 512, 512, 128) == 0    # bm above 256
    assert ws(0, 256, 256, 16, 16) == 0


def test_select_kernel_is_deterministic_and_monotone(lib):
    sel = stof.stof_select_kernel
    assert sel(0.17, 256, 64) == sel(0.17, 256, 64)
    # invalid input -> block-wise
    assert sel(-0.1, 256, 64) == stof.STOF_KERNEL_BLOCKWISE
    assert sel(float("nan"), 256, 64) == stof.STOF_KERNEL_BLOCKWISE
    assert sel(0.5, 0, 64) == stof.STOF_KERNEL_BLOCKWISE
    # denser masks never flip the choice back to row-wise
    for L in (256, 1024, 4096, 16384):
        seen_block = False
        for i in range(101):
            k = sel(i / 100, L, 64)
            if k == stof.STOF_KERNEL_BLOCKWISE:
                seen_block = True
            else:
                assert not seen_block
    assert sel(1.0, 4096, 128) == stof.STOF_KERNEL_BLOCKWISE


FAKE = 1 << 20  # never dereferenced: every call below fails validation first


def _encode(lib, **kw):
    a = dict(mask=FAKE, n_masks=1, lq=256, lk=256, bm=128, bn=128, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    fmt = stof.stof_format()
    return lib.stof_encode_mask(a["mask"], a["n_masks"], a["lq"], a["lk"], a["bm"], a["bn"],
                                a["ws"], a["ws_bytes"], ctypes.byref(fmt), None)


def test_encode_rejects_bad_arguments(lib):
    assert _encode(lib, mask=None) == stof.STOF_ERR_INVALID_ARG
    assert _encode(lib, ws=None) == stof.STOF_ERR_INVALID_ARG
    assert _encode(lib, n_masks=0) == stof.STOF_ERR_INVALID_ARG
    assert _encode(lib, lk=0) == stof.STOF_ERR_INVALID_ARG
    assert _encode(lib, bm=12) == stof.STOF_ERR_SHAPE
    assert _encode(lib, bn=512) == stof.STOF_ERR_SHAPE
    assert _encode(lib, mask=FAKE + 4) == stof.STOF_ERR_ALIGNMENT
    assert _encode(lib, ws=FAKE + 128) == stof.STOF_ERR_ALIGNMENT
    assert _encode(lib, ws_bytes=1000) == stof.STOF_ERR_WORKSPACE
    assert lib.stof_encode_mask(FAKE, 1, 256, 256, 128, 128, FAKE, 1 << 30, None, None) == \
        stof.STOF_ERR_INVALID_ARG


def _fake_format(L=256, bm=128, bn=128, n_masks=1, synced=0):
    f = stof.stof_format()
    f.n_masks, f.lq, f.lk, f.bm, f.bn = n_masks, L, L, bm, bn
    f.n_tr, f.n_tc = L // bm, L // bn
    for name in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "bitmaps",
                 "counts_dev", "scratch"):
        setattr(f, name, FAKE)
    f.synced = synced
    return f


def _mha(lib, fmt=None, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=stof.STOF_BF16, B=1, H=2, L=256, d=64, scale=0.125,
             sb=0, sh=0, which=stof.STOF_KERNEL_ROWWISE, o=FAKE)
    a.update(kw)
    fmt = fmt if fmt is not None else _fake_format()
    return lib.stof_mha_fwd(a["q"], a["k"], a["v"], a["dt"], a["B"], a["H"], a["L"], a["d"],
                            a["scale"], ctypes.byref(fmt), a["sb"], a["sh"], a["which"], a["o"], None)


def test_mha_rejects_bad_arguments(lib):
    assert _mha(lib, q=None) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, o=None) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, dt=7) == stof.STOF_ERR_DTYPE
    assert _mha(lib, which=5) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, B=0) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, scale=float("inf")) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, sb=-1) == stof.STOF_ERR_INVALID_ARG
    assert _mha(lib, d=96) == stof.STOF_ERR_UNSUPPORTED
    assert _mha(lib, L=512) == stof.STOF_ERR_SHAPE                 # format is for L = 256
    assert _mha(lib, sh=1) == stof.STOF_ERR_SHAPE                  # head 1 -> mask 1 of 1
    assert _mha(lib, q=FAKE + 8) == stof.STOF_ERR_ALIGNMENT
    assert _mha(lib, which=stof.STOF_KERNEL_AUTO) == stof.STOF_ERR_NOT_SYNCED
    assert _mha(lib, fmt=_fake_format(bm=64, bn=64), which=stof.STOF_KERNEL_BLOCKWISE) == \
        stof.STOF_ERR_UNSUPPORTED
    f = _fake_format()
    f.bitmaps = None
    assert _mha(lib, fmt=f) == stof.STOF_ERR_INVALID_ARG
    assert lib.stof_format_sync(None, None) == stof.STOF_ERR_INVALID_ARG


def test_binding_checks_shapes_before_calling(lib):
    import torch
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 2, 256, 32, dtype=torch.bfloat16)
    with pytest.raises(stof.StofError):
        stof.stof_mha_fwd(q, q, q, _fake_format(), 0.1, 0, 0, 0, o, stream=0)
    with pytest.raises(stof.StofError):
        stof.stof_mha_fwd(q.float(), q.float(), q.float(), _fake_format(), 0.1, 0, 0, 0, q.float(),
                          stream=0)


def test_binding_checks_new_entry_points_before_calling(lib):
    import torch
    with pytest.raises(stof.StofError):        # last axis must be lk / 8
        stof.stof_encode_mask_bits(torch.zeros(1, 64, 7, dtype=torch.uint8), 64, 16, 16,
                                   torch.zeros(16, dtype=torch.uint8))
    o = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    w = torch.zeros(256, 128, dtype=torch.bfloat16)
    y = torch.zeros(1, 128, 256, dtype=torch.bfloat16)
    with pytest.raises(stof.StofError):        # w must be [N, H*d]
        stof.stof_oproj_fwd(o, torch.zeros(256, 64, dtype=torch.bfloat16), None, None, y)
    with pytest.raises(stof.StofError):        # bias must be [N]
        stof.stof_oproj_fwd(o, w, torch.zeros(128, dtype=torch.bfloat16), None, y)
    with pytest.raises(stof.StofError):        # dtypes must agree
        stof.stof_oproj_fwd(o, w.float(), None, None, y)


def test_oproj_rejects_bad_arguments(lib):
    f = lib.stof_oproj_fwd
    one = ctypes.c_void_p(256)
    assert f(None, one, None, None, 0, 1, 2, 128, 64, 256, one, None, None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, one, None, None, 7, 1, 2, 128, 64, 256, one, None, None) == stof.STOF_ERR_DTYPE
    assert f(one, one, None, None, 0, 1, 2, 128, 96, 256, one, None, None) == stof.STOF_ERR_UNSUPPORTED
    assert f(one, one, None, None, 0, 1, 2, 0, 64, 256, one, None, None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, one, None, None, 0, 1, 2, 128, 64, 200, one, None, None) == stof.STOF_ERR_SHAPE
    assert f(ctypes.c_void_p(8), one, None, None, 0, 1, 2, 128, 64, 256, one, None,
             None) == stof.STOF_ERR_ALIGNMENT


def test_tune_cache_host_side(lib):
    b = stof.stof_tune_density_bucket
    assert b(1.0) == 0 and b(0.5) == -2 and b(0.25) == -4
    assert b(0.7) == -1                      # 2 log2(0.7) = -1.03
    assert b(0.0) == -61 and b(1e-30) == -60
    stof.stof_tune_clear()
    assert stof.stof_tune_lookup(16384, 128, 0.05) is None
    assert stof.stof_tune_workspace_bytes(32, 16384) == max(
        stof.stof_encode_workspace_bytes(32, 16384, 16384, 128, bn) for bn in (64, 128))
    assert stof.stof_tune_workspace_bytes(1, 100) == stof.stof_tune_workspace_bytes(1, 128)  # padded to a tile
    assert stof.stof_tune_workspace_bytes(0, 128) == 0


def test_tune_rejects_bad_arguments(lib):
    res = stof.stof_tune_result()
    st = lib.stof_tune(None, 1, None, None, None, 0, 1, 1, 128, 64, 0.125, 0, 0, None, 0, None,
                       ctypes.byref(res), None)
    assert st == stof.STOF_ERR_INVALID_ARG
    one = ctypes.c_void_p(16)
    st = lib.stof_tune(one, 1, one, one, one, 0, 1, 1, 128, 64, 0.125, 0, 0, one, 16, one,
                       ctypes.byref(res), None)
    assert st == stof.STOF_ERR_WORKSPACE


def test_encode_bits_rejects_bad_arguments(lib):
    fmt = stof.stof_format()
    one = ctypes.c_void_p(256)
    f = lib.stof_encode_mask_bits
    assert f(None, 1, 256, 256, 128, 128, one, 1 << 30, ctypes.byref(fmt), None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, 1, 256, 250, 128, 128, one, 1 << 30, ctypes.byref(fmt), None) == stof.STOF_ERR_SHAPE
    assert f(ctypes.c_void_p(257), 1, 256, 256, 128, 128, one, 1 << 30, ctypes.byref(fmt),
             None) == stof.STOF_ERR_ALIGNMENT
    assert f(one, 1, 256, 256, 128, 128, one, 16, ctypes.byref(fmt), None) == stof.STOF_ERR_WORKSPACE


def test_encode_rules_rejects_bad_arguments(lib):
    fmt = stof.stof_format()
    ws = ctypes.c_void_p(256)
    f = lib.stof_encode_rules

    def call(rules, n=1, lq=256, lk=256, bm=128, bn=128, wsp=ws, ws_bytes=1 << 30, out=ctypes.byref(fmt)):
        return f(rules, n, lq, lk, bm, bn, wsp, ws_bytes, out, None)

    one = (stof.stof_mask_rule * 1)(stof.stof_mask_rule(0, 47, None, None, None, 0))
    assert call(None) == stof.STOF_ERR_INVALID_ARG
    assert call(one, wsp=None) == stof.STOF_ERR_INVALID_ARG
    assert call(one, out=None) == stof.STOF_ERR_INVALID_ARG
    assert call(one, n=0) == stof.STOF_ERR_INVALID_ARG
    many = (stof.stof_mask_rule * 65)()
    assert call(many, n=65) == stof.STOF_ERR_UNSUPPORTED
    blocks_ragged = (stof.stof_mask_rule * 1)(stof.stof_mask_rule(1, 0, None, None, 256, 8))
    assert call(blocks_ragged, lq=250) == stof.STOF_ERR_SHAPE         # a block pattern needs whole blocks
    bad_block = (stof.stof_mask_rule * 1)(stof.stof_mask_rule(1, 0, None, None, 256, 12))
    assert call(bad_block) == stof.STOF_ERR_SHAPE                     # block not a multiple of 8
    bad_block[0].block = 96
    assert call(bad_block) == stof.STOF_ERR_SHAPE                     # 96 does not divide 256
    misaligned = (stof.stof_mask_rule * 1)(stof.stof_mask_rule(1, 0, 258, None, None, 0))
    assert call(misaligned) == stof.STOF_ERR_ALIGNMENT
    assert call(one, wsp=ctypes.c_void_p(128)) == stof.STOF_ERR_ALIGNMENT
    assert call(one, ws_bytes=16) == stof.STOF_ERR_WORKSPACE
    assert ctypes.sizeof(stof.stof_mask_rule) == 40                   # int32 x 2, 3 pointers, int32 + pad


def test_bounded_wait_check_rejects_bad_arguments(lib):
    f = lib.stof_check_bounded_wait
    one = ctypes.c_void_p(256)
    assert f(None, ctypes.c_double(0.1), None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, ctypes.c_double(0.0), None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, ctypes.c_double(11.0), None) == stof.STOF_ERR_INVALID_ARG
    assert f(one, ctypes.c_double(float("nan")), None) == stof.STOF_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(260), ctypes.c_double(0.1), None) == stof.STOF_ERR_ALIGNMENT


def test_missing_library_fails_loudly():
    # no silent fallback: without the built library the binding raises
    code = ("import sys; from sparse_mask_transformer_gb300 import stof\n"
            "try:\n    stof.load_library('/nonexistent/libstof.so')\n"
            "except RuntimeError as e:\n    print('raised', 'missing' in str(e))\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == "raised True", r.stdout + r.stderr


def test_product_package_does_not_import_the_oracle(lib):
    # the oracle is test infrastructure: the package and its binding never load it
    code = ("import sys; import sparse_mask_transformer_gb300 as p; from sparse_mask_transformer_gb300 import stof, synth\n"
            "stof.load_library(); print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == "False", r.stdout + r.stderr


def test_oracle_and_product_share_no_code():
    # the C oracle includes system headers only, and no product source
    # imports, includes or links it
    src = open(os.path.join(ROOT, "oracle", "stof_oracle.c")).read()
    assert not re.search(r'#include\s+"', src)
    for d in ("sparse_mask_transformer_gb300", "include"):
        for dirpath, _, files in os.walk(os.path.join(ROOT, d)):
            for f in files:
                if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                    text = open(os.path.join(dirpath, f)).read()
                    assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                    assert "stof_oracle" not in text, f


def _plan_format(L=1024, bm=128, bn=128, n_masks=1, synced=True, nnz=None, tiles=None):
    """A format struct with non-null (never dereferenced) pointers: the plan
    is host arithmetic on the sizes and the synced counts."""
    f = stof.stof_format()
    f.n_masks, f.lq, f.lk, f.bm, f.bn = n_masks, L, L, bm, bn
    f.n_tr, f.n_tc = L // bm, L // bn
    for name in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "bitmaps", "counts_dev",
                 "scratch"):
        setattr(f, name, 1 << 20)
    f.synced = 1 if synced else 0
    f.nnz = nnz if nnz is not None else L * L // 2
    f.n_full = 0
    f.n_part = tiles if tiles is not None else f.n_tr * f.n_tc // 2
    return f


def test_mha_plan_sources_and_variants(lib):
    stof.stof_tune_clear()
    f = _plan_format()
    p = stof.stof_mha_plan(f, 1, 4, 1024, 64, stof.STOF_KERNEL_ROWWISE)
    assert (p.kernel, p.stages, p.persistent, p.source) == (stof.STOF_KERNEL_ROWWISE, 0, 0, stof.STOF_PLAN_FORCED)
    assert p.rows_per_warp == 1                                      # 512 keys per row: a warp each
    assert stof.stof_mha_plan(_plan_format(nnz=20 * 1024), 1, 2, 1024, 64, 0).rows_per_warp == 1  # 2048 rows
    # more rows: rows per warp by the mean valid keys per row
    assert stof.stof_mha_plan(_plan_format(nnz=20 * 1024), 1, 64, 1024, 64, 0).rows_per_warp == 4
    assert stof.stof_mha_plan(_plan_format(nnz=100 * 1024), 1, 64, 1024, 64, 0).rows_per_warp == 2
    # few keys on average but many per listed OT (keys in blocks): one row per warp
    assert stof.stof_mha_plan(_plan_format(nnz=20 * 1024, tiles=2), 1, 64, 1024, 64, 0).rows_per_warp == 1
    assert stof.stof_mha_plan(_plan_format(nnz=512 * 1024), 1, 64, 1024, 64, 0).rows_per_warp == 1
    assert stof.stof_mha_plan(_plan_format(nnz=20 * 1024, synced=False), 1, 64, 1024, 64, 0).rows_per_warp == 1
    p = stof.stof_mha_plan(f, 1, 4, 1024, 64, stof.STOF_KERNEL_BLOCKWISE)
    # 32 of 64 OTs listed over 8 OT rows: 4 per row, below the persistent threshold at d = 64
    assert (p.kernel, p.persistent, p.stages, p.source) == (stof.STOF_KERNEL_BLOCKWISE, 1, 4, stof.STOF_PLAN_FORCED)
    p = stof.stof_mha_plan(f, 1, 4, 1024, 128, stof.STOF_KERNEL_BLOCKWISE)
    assert (p.persistent, p.stages) == (0, 3)                       # d = 128: one CTA per query tile
    p = stof.stof_mha_plan(_plan_format(L=16384, tiles=128 * 100), 1, 1, 16384, 64, stof.STOF_KERNEL_BLOCKWISE)
    assert (p.persistent, p.stages) == (0, 3)                       # 100 OTs per row: one CTA per query tile
    p = stof.stof_mha_plan(f, 1, 4, 1024, 64, stof.STOF_KERNEL_AUTO)
    assert p.source == stof.STOF_PLAN_ANALYTIC
    assert p.kernel == stof.stof_select_kernel(0.5, 1024, 64)


def test_mha_plan_rejects_what_the_call_rejects(lib):
    f = _plan_format()
    with pytest.raises(stof.StofError) as e:
        stof.stof_mha_plan(_plan_format(synced=False), 1, 1, 1024, 64, stof.STOF_KERNEL_AUTO)
    assert e.value.status == stof.STOF_ERR_NOT_SYNCED
    with pytest.raises(stof.StofError) as e:
        stof.stof_mha_plan(_plan_format(bm=64, bn=64), 1, 1, 1024, 64, stof.STOF_KERNEL_BLOCKWISE)
    assert e.value.status == stof.STOF_ERR_UNSUPPORTED
    # AUTO on OTs the block-wise kernel does not take falls back to the row-wise kernel
    p = stof.stof_mha_plan(_plan_format(bm=64, bn=64, nnz=1024 * 1024), 1, 1, 1024, 64, stof.STOF_KERNEL_AUTO)
    assert p.kernel == stof.STOF_KERNEL_ROWWISE
    for args, status in [((1, 1, 2048, 64, 0), stof.STOF_ERR_SHAPE),      # L differs from the format's
                         ((1, 1, 1024, 96, 0), stof.STOF_ERR_UNSUPPORTED),
                         ((0, 1, 1024, 64, 0), stof.STOF_ERR_INVALID_ARG),
                         ((1, 1, 1024, 64, 7), stof.STOF_ERR_INVALID_ARG)]:
        with pytest.raises(stof.StofError) as e:
            stof.stof_mha_plan(f, *args)
        assert e.value.status == status, args
    assert lib.stof_mha_plan(ctypes.byref(f), 1, 1, 1024, 64, 0, None) == stof.STOF_ERR_INVALID_ARG


def test_python_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors against the C compiler's layout of the
    header's structs (sizes and every field offset)."""
    structs = {"stof_format": stof.stof_format, "stof_plan": stof.stof_plan,
               "stof_tune_result": stof.stof_tune_result, "stof_mask_rule": stof.stof_mask_rule}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "stof.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe)])
    got = dict(ln.split() for ln in subprocess.check_output([str(exe)], text=True).splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(got[f"{name}.{field}"]) == getattr(cls, field).offset, (name, field)


def test_select_kernel_heads_model(lib):
    sel = stof.stof_select_kernel_heads
    row, blk = stof.STOF_KERNEL_ROWWISE, stof.STOF_KERNEL_BLOCKWISE
    # the window-48 workload (2 heads, L = 256, 3 partial OTs over 2 query tiles) is row-wise territory
    assert sel(0.1703, 256, 64, 2, 3 / 2) == row
    # the other workloads are block-wise
    assert sel(0.969, 512, 64, 16 * 12, 4.0) == blk
    assert sel(0.5002, 2048, 64, 8 * 12, 136 / 16) == blk
    assert sel(0.135, 4096, 64, 4 * 16, 884 / 32) == blk
    assert sel(0.0501, 16384, 128, 32, 8256 / 128) == blk
    # more heads never turn a block-wise choice into a row-wise one
    for rho in (0.01, 0.05, 0.2):
        for L in (128, 512, 2048):
            ks = [sel(rho, L, 64, h, -1) for h in (1, 2, 4, 16, 64, 256, 4096)]
            assert ks == sorted(ks), (rho, L, ks)   # ROWWISE (0) before BLOCKWISE (1)
    # one head, every OT listed: the three-argument form
    for rho in (0.0, 0.05, 0.5):
        assert stof.stof_select_kernel(rho, 1024, 128) == sel(rho, 1024, 128, 1, -1)
    assert sel(0.1, 1024, 64, 0, -1) == blk       # invalid head count


def _plan_call(lib, plan, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=stof.STOF_BF16, B=1, H=2, L=256, d=64, scale=0.125, sb=0, sh=0, o=FAKE)
    a.update(kw)
    fmt = _fake_format()
    return lib.stof_mha_fwd_plan(a["q"], a["k"], a["v"], a["dt"], a["B"], a["H"], a["L"], a["d"], a["scale"],
                                 ctypes.byref(fmt), a["sb"], a["sh"], None if plan is None else ctypes.byref(plan),
                                 a["o"], None)


def test_mha_fwd_plan_rejects_bad_plans_before_launch(lib):
    P = stof.stof_plan
    assert _plan_call(lib, None) == stof.STOF_ERR_INVALID_ARG
    assert _plan_call(lib, P(5, 0, 0, 0, 0)) == stof.STOF_ERR_INVALID_ARG              # unknown kernel
    assert _plan_call(lib, P(stof.STOF_KERNEL_AUTO, 0, 0, 0, 0)) == stof.STOF_ERR_INVALID_ARG
    assert _plan_call(lib, P(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 3)) == stof.STOF_ERR_UNSUPPORTED  # rows per warp
    assert _plan_call(lib, P(stof.STOF_KERNEL_BLOCKWISE, 9, 0, 0, 0)) == stof.STOF_ERR_INVALID_ARG
    assert _plan_call(lib, P(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 1), q=None) == stof.STOF_ERR_INVALID_ARG
    assert _plan_call(lib, P(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 1), d=96) == stof.STOF_ERR_UNSUPPORTED
    blk = stof.STOF_KERNEL_BLOCKWISE
    assert _plan_call(lib, P(blk, 0, 1, 0, 0, 2, 0)) == stof.STOF_ERR_INVALID_ARG        # exp split is 0 or 1
    assert _plan_call(lib, P(blk, 0, 1, 0, 0, 0, 3)) == stof.STOF_ERR_UNSUPPORTED        # 2 or 4 warpgroups
    assert _plan_call(lib, P(blk, 0, 1, 0, 0, 0, 8)) == stof.STOF_ERR_UNSUPPORTED
    assert _plan_call(lib, P(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 1, 1, 0)) == stof.STOF_ERR_UNSUPPORTED
    assert _plan_call(lib, P(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 1, 0, 4)) == stof.STOF_ERR_UNSUPPORTED


def test_oproj_ln_sizes_and_argument_errors(lib):
    assert stof.stof_oproj_ln_workspace_bytes(2, 256, 512) == 2 * 256 * 2 * 8
    assert stof.stof_oproj_ln_workspace_bytes(1, 128, 300) == 0      # N not a multiple of 256
    assert stof.stof_oproj_ln_workspace_bytes(0, 128, 256) == 0

    def call(**kw):
        a = dict(o=FAKE, w=FAKE, bias=None, res=None, gamma=None, beta=None, eps=1e-5, dt=stof.STOF_BF16, B=1, H=2,
                 L=128, d=64, N=256, y=FAKE, ws=FAKE, ws_bytes=1 << 20)
        a.update(kw)
        return lib.stof_oproj_ln_fwd(a["o"], a["w"], a["bias"], a["res"], a["gamma"], a["beta"], a["eps"], a["dt"],
                                     a["B"], a["H"], a["L"], a["d"], a["N"], a["y"], a["ws"], a["ws_bytes"], None,
                                     None)
    assert call(o=None) == stof.STOF_ERR_INVALID_ARG
    assert call(ws=None) == stof.STOF_ERR_INVALID_ARG
    assert call(eps=0.0) == stof.STOF_ERR_INVALID_ARG
    assert call(eps=float("inf")) == stof.STOF_ERR_INVALID_ARG
    assert call(ws_bytes=100) == stof.STOF_ERR_WORKSPACE
    assert call(gamma=FAKE + 4) == stof.STOF_ERR_ALIGNMENT
    assert call(N=300) == stof.STOF_ERR_SHAPE
    assert call(d=96) == stof.STOF_ERR_UNSUPPORTED
    assert call(dt=5) == stof.STOF_ERR_DTYPE


def test_head_dims_outside_the_block_wise_kernels_plan_row_wise(lib):
    """d = 32 and 256 are the row-wise kernel's alone: AUTO plans it (at most
    2 query rows per warp at d = 256, whose key needs 16 lanes), and a forced
    block-wise call is refused before any launch."""
    for d in (32, 256):
        p = stof.stof_mha_plan(_plan_format(L=1024, nnz=1024 * 1024), 1, 64, 1024, d, stof.STOF_KERNEL_AUTO)
        assert p.kernel == stof.STOF_KERNEL_ROWWISE
        assert p.rows_per_warp in ((1, 2, 4) if d == 32 else (1, 2))
        with pytest.raises(stof.StofError) as e:
            stof.stof_mha_plan(_plan_format(L=1024), 1, 1, 1024, d, stof.STOF_KERNEL_BLOCKWISE)
        assert e.value.status == stof.STOF_ERR_UNSUPPORTED
    few = stof.stof_mha_plan(_plan_format(L=1024, nnz=20 * 1024), 1, 64, 1024, 256, stof.STOF_KERNEL_AUTO)
    assert few.rows_per_warp <= 2


def test_binding_refuses_a_host_mask_that_is_not_pinned():
    """A host mask is only readable by the device from pinned memory; the
    binding refuses any other before it calls the library."""
    import torch
    mask = torch.zeros(1, 128, 128, dtype=torch.uint8)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(stof.StofError) as e:
        stof.stof_encode_mask(mask, 128, 128, ws)
    assert e.value.status == stof.STOF_ERR_INVALID_ARG
