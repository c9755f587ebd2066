"""The C-ABI library loads and exports what include/*.h declares; argument
checks that run before any launch answer correctly without a GPU."""

import ctypes
import glob
import os
import re

import pytest

import paged_kv_cache_288_gb300 as pa
from paged_kv_cache_288_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return pa.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?(pa_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for f in ("pa_reshape_and_cache", "pa_decode", "pa_decode_workspace_size", "pa_copy_blocks",
              "pa_swap_blocks",
              "pa_status_string", "pa_last_error_message", "pa_version"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    assert pa.lib().pa_status_string(0) == b"PA_OK"
    assert pa.lib().pa_status_string(4) == b"PA_ERR_WORKSPACE"
    assert L.pa_version() >= 100


NULL = None


def _decode(L, **kw):
    args = dict(out=16, q=16, k=16, v=16, tables=16, width=16, lens=16, B=2, Hq=8, Hkv=2, d=128,
                bs=16, Nb=100, scale=0.1, qt=pa.BF16, kvt=pa.BF16, ks=NULL, vs=NULL, maxctx=100,
                part=0, ws=NULL, wsb=0, err=NULL, stream=NULL)
    args.update(kw)
    return L.pa_decode(args["out"], args["q"], args["k"], args["v"], args["tables"], args["width"],
                       args["lens"], args["B"], args["Hq"], args["Hkv"], args["d"], args["bs"],
                       args["Nb"], args["scale"], args["qt"], args["kvt"], args["ks"], args["vs"],
                       args["maxctx"], args["part"], args["ws"], args["wsb"], args["err"],
                       args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),                 # heads not a multiple
    (dict(d=100), 1),                      # head_dim not a multiple of 8
    (dict(bs=12), 2),                      # unsupported block size
    (dict(Hq=48, Hkv=4), 2),               # group of 12
    (dict(d=96), 2),                       # unsupported head_dim
    (dict(qt=pa.F16), 1),                  # q and cache types differ
    (dict(kvt=pa.FP8_E4M3), 1),            # fp8 without scales
    (dict(qt=pa.FP8_E4M3), 1),             # fp8 queries
    (dict(maxctx=16 * 16 + 1), 1),         # above table width * block size
    (dict(part=24), 1),                    # partition not a multiple of 16
    (dict(part=32, bs=64), 1),             # partition not a multiple of the block size
    (dict(part=64, ws=NULL), 4),           # split path without workspace
    (dict(scale=float("inf")), 1),
    (dict(out=NULL), 1),
    (dict(q=24), 1),                       # misaligned
    (dict(ws=64, wsb=1 << 20, part=64), 1),  # workspace not 256-byte aligned
    (dict(B=-1), 1),
    (dict(B=0), 0),                        # nothing to do
])
def test_decode_argument_checks(L, kw, status):
    assert _decode(L, **kw) == status, pa.lib().pa_last_error_message()


def test_reshape_and_cache_argument_checks(L):
    f = L.pa_reshape_and_cache
    ok = (16, 16, 16, 16, 16, 4, 2, 128, 16, 10, pa.F16, pa.F16, NULL, NULL, NULL, NULL)
    bad = list(ok)
    bad[7] = 12
    assert f(*bad) == 1  # head_dim
    bad = list(ok)
    bad[11] = pa.BF16
    assert f(*bad) == 1  # source and 16-bit cache types differ
    bad = list(ok)
    bad[11] = pa.FP8_E4M3
    assert f(*bad) == 1  # fp8 without scales
    bad = list(ok)
    bad[0] = 8
    assert f(*bad) == 1  # misaligned
    bad = list(ok)
    bad[5] = 0
    assert f(*bad) == 0  # no tokens


def test_copy_blocks_argument_checks(L):
    f = L.pa_copy_blocks
    assert f(16, 16, 2, 16, 3, 10, 100, NULL, NULL) == 1      # block_bytes not a multiple of 16
    assert f(16, 16, 2, 16, 3, 0, 128, NULL, NULL) == 1       # no blocks
    assert f(16, 16, 0, 16, 3, 10, 128, NULL, NULL) == 0      # no layers: nothing to do
    assert f(NULL, 16, 2, 16, 3, 10, 128, NULL, NULL) == 1


def test_workspace_size(L):
    assert pa.decode_workspace_size(64, 32, 8, 128, 4096, 512) > 64 * 32 * 8 * 128 * 4
    assert pa.decode_workspace_size(4, 4, 2, 64, 64, 0) >= 0
    assert pa.decode_workspace_size(0, 4, 2, 64, 64, 0) == 0


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_288_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        src = open(path).read()
        assert not re.search(r"^\s*(from|import)\s+oracle", src, flags=re.M), path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        src = open(path).read()
        assert "paged_kv_cache_288_gb300" not in src and "workloads" not in src, path


def test_swap_blocks_argument_checks(L):
    arr = (ctypes.c_void_p * 65)(*([16] * 65))
    def swap(layers=1, pairs=1, snb=4, dnb=4, bb=4096):
        return L.pa_swap_blocks(arr, arr, arr, arr, layers, 16, pairs, snb, dnb, bb, NULL, NULL)
    assert swap(layers=65) == 2           # PA_ERR_UNSUPPORTED: over PA_SWAP_MAX_LAYERS
    assert swap(layers=-1) == 1           # PA_ERR_INVALID
    assert swap(pairs=-1) == 1
    assert swap(snb=0) == 1
    assert swap(bb=4000) == 1             # not a multiple of 16
    assert swap(pairs=0) == 0             # nothing to move: no CUDA call
    assert swap(layers=0) == 0
    assert L.pa_swap_blocks(None, arr, arr, arr, 1, 16, 1, 4, 4, 4096, NULL, NULL) == 1


def _prefill(L, **kw):
    args = dict(out=16, q=16, k=16, v=16, tables=16, width=16, lens=16, qstart=16, B=2, T=64, maxq=32,
                Hq=32, Hkv=8, d=128, bs=16, Nb=100, scale=0.1, dt=pa.BF16, err=NULL, stream=NULL)
    args.update(kw)
    return L.pa_prefill(args["out"], args["q"], args["k"], args["v"], args["tables"], args["width"],
                        args["lens"], args["qstart"], args["B"], args["T"], args["maxq"], args["Hq"],
                        args["Hkv"], args["d"], args["bs"], args["Nb"], args["scale"], args["dt"],
                        args["err"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),                # heads not a multiple
    (dict(bs=12), 2),                      # unsupported block size
    (dict(d=64), 2),                       # head_dim 128 only
    (dict(Hq=24, Hkv=8), 2),               # group of 3
    (dict(dt=pa.FP8_E4M3), 2),             # 16-bit only
    (dict(Nb=0), 1),                       # empty pool
    (dict(B=-1), 1),
    (dict(out=NULL), 1),
    (dict(q=24), 1),                       # misaligned
    (dict(B=70000), 2),                    # more sequences than the grid takes
    (dict(B=0), 0),                        # nothing to do
    (dict(maxq=0), 0),
])
def test_prefill_argument_checks(L, kw, status):
    assert _prefill(L, **kw) == status, pa.lib().pa_last_error_message()


def _noalloc(L, **kw):
    args = dict(out=16, q=16, k=16, v=16, tables=16, width=1024, lens=16, B=256, Hq=64, Hkv=8,
                d=128, bs=16, Nb=100, scale=0.1, qt=pa.BF16, kvt=pa.BF16, maxctx=16384, part=512,
                err=NULL, stream=NULL)
    args.update(kw)
    return L.pa_decode_split_noalloc(
        args["out"], args["q"], args["k"], args["v"], args["tables"], args["width"], args["lens"],
        args["B"], args["Hq"], args["Hkv"], args["d"], args["bs"], args["Nb"], args["scale"],
        args["qt"], args["kvt"], NULL, NULL, args["maxctx"], args["part"], args["err"],
        args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(part=-16), 1),                   # negative partition size: invalid, not 512
    (dict(Hq=6, Hkv=4), 1),                # a bad argument is reported before the size
    (dict(d=100), 1),
    (dict(bs=12, part=48, maxctx=12000), 2),
    (dict(out=NULL), 1),
    (dict(), 4),                           # valid, but the partials exceed the scratch
    (dict(B=0), 0),                        # nothing to do
])
def test_noalloc_argument_checks(L, kw, status):
    assert _noalloc(L, **kw) == status, pa.lib().pa_last_error_message()


def test_binding_refuses_host_tensors():
    """The binding hands raw pointers to the C ABI, so it refuses tensors the
    kernels could not read as dense device memory (before loading anything)."""
    import torch
    q = torch.zeros(2, 8, 64, dtype=torch.float16)
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16)
    tables = torch.zeros(2, 4, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        pa.decode(torch.empty_like(q), q, kc, kc, tables, lens, 0.1, 16)
    key = torch.zeros(3, 2, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.reshape_and_cache(key, key, kc, kc, torch.zeros(3, dtype=torch.int64))
    qs = torch.tensor([0, 1, 2], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.prefill(torch.empty_like(q), q, kc, kc, tables, lens, qs, 0.1, 1)
    ptrs = torch.zeros(1, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.copy_blocks(ptrs, ptrs, torch.zeros(1, 2, dtype=torch.int64), 4, 4096)


def _shared(L, **kw):
    args = dict(out=16, q=16, k=16, v=16, tables=16, width=16, lens=16, B=4, Hq=8, Hkv=2, d=128,
                bs=16, Nb=100, scale=0.1, dt=pa.BF16, maxctx=100, gs=16, gp=16, ng=1, mgs=4, mpl=64,
                ws=256, wsb=1 << 20, err=NULL, stream=NULL)
    args.update(kw)
    return L.pa_decode_shared_prefix(
        args["out"], args["q"], args["k"], args["v"], args["tables"], args["width"], args["lens"],
        args["B"], args["Hq"], args["Hkv"], args["d"], args["bs"], args["Nb"], args["scale"],
        args["dt"], args["maxctx"], args["gs"], args["gp"], args["ng"], args["mgs"], args["mpl"],
        args["ws"], args["wsb"], args["err"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dt=pa.FP8_E4M3), 1),             # 16-bit caches only (q must be 16-bit)
    (dict(d=256), 2),
    (dict(Hq=12, Hkv=1), 2),               # group of 12
    (dict(ng=-1), 1),
    (dict(mpl=-16), 1),
    (dict(gs=NULL), 1),                    # groups without their arrays
    (dict(ws=NULL), 1),
    (dict(ws=128), 1),                     # workspace not 256-byte aligned
    (dict(B=3000), 2),                     # more sequences than the tensor-core schedule takes
    (dict(B=0), 0),
])
def test_shared_prefix_argument_checks(L, kw, status):
    assert _shared(L, **kw) == status, pa.lib().pa_last_error_message()
