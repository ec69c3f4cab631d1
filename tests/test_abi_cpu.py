"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every entry point include/minisgl.h declares, and rejects bad
arguments with the documented error codes before any device work."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_row_gb300 import build
    build.build()
    import paged_kv_cache_row_gb300 as p
    return p.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "minisgl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(minisgl_\w+)\s*\(", text)))


def test_header_declares_the_path():
    syms = declared_symbols()
    for s in ("minisgl_store_kv", "minisgl_decode_attn", "minisgl_extend_attn"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    import paged_kv_cache_row_gb300 as p
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} declared in minisgl.h but not exported"
    assert sorted(p.EXPORTED_SYMBOLS) == declared_symbols()


def test_check_indices_rejects_bad_arguments_on_host(lib):
    fake = 1 << 40  # never dereferenced: validation fails before any device work
    assert lib.minisgl_check_indices(fake, 4, 32, 32, fake, fake, 4, 100, None, None) == -1
    assert b"counts" in lib.minisgl_last_error()
    assert lib.minisgl_check_indices(fake, -1, 32, 32, fake, fake, 4, 100, fake, None) == -1
    assert lib.minisgl_check_indices(fake, 4, 32, 32, fake, fake, 4, 0, fake, None) == -1
    assert lib.minisgl_check_indices(None, 4, 32, 32, fake, fake, 4, 100, fake, None) == -1
    assert lib.minisgl_check_indices(fake, 4, 32, 32, fake, None, 4, 100, fake, None) == -1
    assert lib.minisgl_check_indices(fake, 4, 16, 32, fake, fake, 4, 100, fake, None) == -3


def test_error_codes_on_host(lib):
    import paged_kv_cache_row_gb300 as p
    fake = 1 << 40  # never dereferenced: every call below fails validation first
    d = p._PoolDesc(k_base=fake, v_base=fake, layer_stride=8 * 100 * 128, row_stride=8 * 128,
                    num_layers=1, num_rows=100, num_kv_heads=8, head_dim=128, page_size=1,
                    dtype=p.MINISGL_BF16)
    ref = ctypes.byref
    # NULL pool
    assert lib.minisgl_store_kv(None, 0, fake, fake, 1024, 1024, fake, 4, None) == -1
    # bad layer
    assert lib.minisgl_store_kv(ref(d), 3, fake, fake, 1024, 1024, fake, 4, None) == -1
    assert b"layer" in lib.minisgl_last_error()
    # token stride below the row
    assert lib.minisgl_store_kv(ref(d), 0, fake, fake, 512, 1024, fake, 4, None) == -3
    # dtype
    bad = p._PoolDesc.from_buffer_copy(d)
    bad.dtype = 7
    assert lib.minisgl_decode_attn(ref(bad), 0, fake, 16, fake, 4, 32, 32, fake, 0.1, fake, fake,
                                   1 << 20, 0, None) == -2
    # head_dim
    bad = p._PoolDesc.from_buffer_copy(d)
    bad.head_dim = 96
    assert lib.minisgl_decode_attn(ref(bad), 0, fake, 16, fake, 4, 32, 32, fake, 0.1, fake, fake,
                                   1 << 20, 0, None) == -4
    # group size 32 > 16, and a non-multiple head count
    assert lib.minisgl_decode_attn(ref(d), 0, fake, 256, fake, 4, 32, 32, fake, 0.1, fake, fake,
                                   1 << 20, 0, None) == -4
    assert lib.minisgl_decode_attn(ref(d), 0, fake, 12, fake, 4, 32, 32, fake, 0.1, fake, fake,
                                   1 << 20, 0, None) == -3
    # workspace too small (needs 2 splits)
    need = lib.minisgl_decode_workspace_bytes(4, 16, 8, 128, 2)
    assert need > 0
    assert lib.minisgl_decode_attn(ref(d), 0, fake, 16, fake, 4, 32, 32, fake, 0.1, fake, fake,
                                   need - 1, 0, None) == -6
    # page table narrower than its width
    assert lib.minisgl_decode_attn(ref(d), 0, fake, 16, fake, 4, 16, 32, fake, 0.1, fake, fake,
                                   need, 0, None) == -3
    # extend: head_dim 96 unsupported, group 17 unsupported, unaligned work counter
    bad = p._PoolDesc.from_buffer_copy(d)
    bad.head_dim = 96
    bad.row_stride = 8 * 96
    assert lib.minisgl_extend_attn(ref(bad), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10,
                                   0.1, fake, None, None) == -4
    d17 = p._PoolDesc.from_buffer_copy(d)
    d17.num_kv_heads = 1
    d17.row_stride = 128
    assert lib.minisgl_extend_attn(ref(d17), 0, fake, 17, fake, 2, 32, 32, fake, fake, fake, 10,
                                   0.1, fake, None, None) == -4
    assert lib.minisgl_extend_attn(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10,
                                   0.1, fake, fake + 4, None) == -1
    # extend needs a positive, finite sm_scale
    assert lib.minisgl_extend_attn(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10,
                                   -0.1, fake, None, None) == -1
    assert lib.minisgl_extend_attn(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10,
                                   float("nan"), fake, None, None) == -1
    # rope_store_kv: q stride below H_q*d, unaligned table, no table rows, NULL positions
    rs = lib.minisgl_rope_store_kv
    assert rs(ref(d), 0, fake, 16, 1024, fake, fake, 1024, 1024, fake, fake, 64, fake, 4, None) == -3
    assert rs(ref(d), 0, fake, 16, 2048, fake, fake, 1024, 1024, fake, fake + 4, 64, fake, 4, None) == -3
    assert rs(ref(d), 0, fake, 16, 2048, fake, fake, 1024, 1024, fake, fake, 0, fake, 4, None) == -1
    assert rs(ref(d), 0, fake, 16, 2048, fake, fake, 1024, 1024, None, fake, 64, fake, 4, None) == -1
    assert rs(ref(d), 0, fake, 0, 2048, fake, fake, 1024, 1024, fake, fake, 64, fake, 4, None) == -1
    assert rs(ref(d), 0, fake, 16, 2048, fake, fake, 1024, 1024, fake, fake, 64, fake, 0, None) == 0
    # cascade decode: shared_len outside [1, width], workspace too small, head_dim 96
    cd = lib.minisgl_cascade_decode_attn
    big = lib.minisgl_cascade_workspace_bytes(4, 16, 8, 128)
    assert big > 0 and lib.minisgl_cascade_workspace_bytes(-1, 16, 8, 128) == 0
    assert cd(ref(d), 0, fake, 16, fake, 4, 32, 32, fake, 0, 0.1, fake, fake, big, None) == -1
    assert cd(ref(d), 0, fake, 16, fake, 4, 32, 32, fake, 33, 0.1, fake, fake, big, None) == -1
    assert cd(ref(d), 0, fake, 16, fake, 4, 32, 32, fake, 16, 0.1, fake, fake, 1024, None) == -6
    assert b"workspace" in lib.minisgl_last_error()
    assert cd(ref(bad), 0, fake, 16, fake, 4, 32, 32, fake, 16, 0.1, fake, fake, big, None) == -4
    # cascade extend: shared_len outside [1, width], workspace too small, head_dim 96
    ce = lib.minisgl_cascade_extend_attn
    cbig = lib.minisgl_cascade_extend_workspace_bytes(10, 16, 128)
    assert cbig == 256 + (10 * 16 * 128 * 4 + 255) // 256 * 256 + (10 * 16 * 4 + 255) // 256 * 256
    assert ce(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10, 0, 0.1, fake, fake, cbig, None) == -1
    assert ce(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10, 33, 0.1, fake, fake, cbig, None) == -1
    assert ce(ref(d), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10, 8, 0.1, fake, fake, cbig - 1,
              None) == -6
    assert ce(ref(bad), 0, fake, 16, fake, 2, 32, 32, fake, fake, fake, 10, 8, 0.1, fake, fake, cbig,
              None) == -4
    # shared-prefix check: NULL counts, shared_len outside [1, width], NULL lens
    cs = lib.minisgl_check_shared_prefix
    assert cs(fake, 4, 32, 32, 8, fake, None, None) == -1
    assert cs(fake, 4, 32, 32, 0, fake, fake, None) == -1
    assert cs(fake, 4, 32, 32, 33, fake, fake, None) == -1
    assert cs(fake, 4, 32, 32, 8, None, fake, None) == -1
    assert cs(fake, 4, 16, 32, 8, fake, fake, None) == -3
    # empty work is a no-op that touches nothing
    assert lib.minisgl_store_kv(ref(d), 0, fake, fake, 1024, 1024, fake, 0, None) == 0
    assert lib.minisgl_decode_attn(ref(d), 0, fake, 16, fake, 0, 32, 32, fake, 0.1, fake, fake,
                                   0, 0, None) == 0


def test_workspace_bytes_formula(lib):
    def al(x):
        return (x + 255) // 256 * 256
    for B, Hq, Hk, d, S in [(4, 8, 2, 64, 2), (64, 16, 8, 128, 16), (256, 32, 8, 128, 17)]:
        want = al(B * Hk * 4) + al(B * Hq * S * 4) + B * Hq * S * d * 4
        assert lib.minisgl_decode_workspace_bytes(B, Hq, Hk, d, S) == want
    assert lib.minisgl_decode_workspace_bytes(4, 8, 2, 64, 1) == 0
    assert lib.minisgl_decode_workspace_bytes(4, 8, 2, 64, 257) == 0


def test_kv_pool_bytes_golden():
    import paged_kv_cache_row_gb300 as p
    fx = json.load(open(os.path.join(ROOT, "tests", "golden", "kv_cache_size_example.json")))
    got = p.kv_pool_bytes(fx["num_layers"], fx["num_kv_heads"], fx["head_dim"], fx["num_tokens"],
                          fx["elem_bytes"])
    assert got == fx["expected_bytes"]


def test_binding_row_check_reads_shapes_and_strides():
    """The binding's check that k / v hold [n, ...] rows of `row` contiguous
    elements agrees with indexing a row and asking torch, on layouts that pass
    and layouts that do not (and accepts zero rows, which indexing cannot)."""
    import torch
    from paged_kv_cache_row_gb300 import _rows_ok

    def by_indexing(t, n, row):
        return t.shape[0] == n and t[0].numel() == row and t[0].is_contiguous()

    cases = [torch.zeros(5, 8, 128),                       # dense
             torch.zeros(5, 2048)[:, :1024],               # rows padded to a wider stride
             torch.zeros(5, 8, 256)[:, :, :128],           # heads padded: rows not contiguous
             torch.zeros(8, 5, 128).transpose(0, 1),       # token and head axes swapped
             torch.zeros(5, 1, 1024),                      # a size-1 axis with any stride
             torch.zeros(5, 128, 8).transpose(1, 2),       # channels strided
             torch.zeros(10, 8, 128)[::2],                 # every other token
             torch.zeros(5, 8, 128, 1),                    # trailing size-1 axis
             torch.zeros(5, 4, 128)]                       # wrong row length
    for t in cases:
        assert _rows_ok(t, 5, 1024) == by_indexing(t, 5, 1024), (tuple(t.shape), t.stride())
        assert not _rows_ok(t, 6, 1024)
    assert _rows_ok(torch.zeros(0, 8, 128), 0, 1024)
    assert not _rows_ok(torch.zeros(1024), 1024, 1)
