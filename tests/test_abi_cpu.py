"""The C ABI on the CPU: the library loads, exports every symbol include/splash.h
declares, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "splash.h")


@pytest.fixture(scope="module")
def splash():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as bsf
    return bsf


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(splash_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("splash_build_mask_info", "splash_attention_fwd", "splash_mask_info_counts",
                     "splash_mask_info_to_host", "splash_mask_info_destroy", "splash_last_device_error",
                     "splash_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(splash):
    lib = splash.lib()
    for name in declared_functions():
        assert hasattr(lib, name), f"libsplash.so does not export {name}"


def test_status_strings_and_version(splash):
    lib = splash.lib()
    for code in range(8):
        s = lib.splash_status_string(code).decode()
        assert s.startswith("SPLASH_")
    assert lib.splash_status_string(99).decode() == "SPLASH_ERR_UNKNOWN"
    assert "sm_103a" in splash.version()


def test_invalid_arguments_are_rejected_before_any_launch(splash):
    lib = splash.lib()
    out = ctypes.c_void_p()
    spec = splash._Spec(1, -1, -1, None, None, 0)
    null = ctypes.c_void_p(0)
    # no output pointer / no spec
    assert lib.splash_build_mask_info(ctypes.byref(spec), 256, 256, 64, 64, null, None) == 1
    assert lib.splash_build_mask_info(None, 256, 256, 64, 64, null, ctypes.byref(out)) == 1
    # bad sizes and unsupported blocks
    assert lib.splash_build_mask_info(ctypes.byref(spec), 0, 256, 64, 64, null, ctypes.byref(out)) == 1
    assert lib.splash_build_mask_info(ctypes.byref(spec), 256, 256, 32, 32, null, ctypes.byref(out)) == 3
    assert lib.splash_build_mask_info(ctypes.byref(spec), 256, 256, 64, 96, null, ctypes.byref(out)) == 3
    # query blocks may be 256 rows tall, key blocks may not
    assert lib.splash_build_mask_info(ctypes.byref(spec), 512, 512, 128, 256, null, ctypes.byref(out)) == 3
    assert lib.splash_build_mask_info(ctypes.byref(spec), 512, 512, 512, 128, null, ctypes.byref(out)) == 3
    bad = splash._Spec(2, -1, -1, None, None, 0)
    assert lib.splash_build_mask_info(ctypes.byref(bad), 256, 256, 64, 64, null, ctypes.byref(out)) == 1
    bad = splash._Spec(1, -5, -1, None, None, 0)
    assert lib.splash_build_mask_info(ctypes.byref(bad), 256, 256, 64, 64, null, ctypes.byref(out)) == 1
    segs = splash._Spec(1, -1, -1, 16, None, 0)   # segment pointer with batch 0
    assert lib.splash_build_mask_info(ctypes.byref(segs), 256, 256, 64, 64, null, ctypes.byref(out)) == 1
    assert not out
    # attention: NULL tensors / handle
    f = lib.splash_attention_fwd
    assert f(None, None, None, 1, 2, 2, 256, 256, 64, 64, None, None, None, 0.125, 0.0, None, None, null) == 1
    # non-positive / NaN scale (checked before the handle is touched)
    fake = ctypes.c_void_p(16)
    assert f(fake, fake, fake, 1, 2, 2, 256, 256, 64, 64, None, None, fake, 0.0, 0.0, fake, fake, null) == 1
    assert f(fake, fake, fake, 1, 2, 2, 256, 256, 64, 64, None, None, fake, float("nan"), 0.0, fake, fake, null) == 1
    # the Max Logit Estimate variant and the backward: NULL tensors, bad scale
    fm = lib.splash_attention_fwd_mle
    assert fm(None, None, None, 1, 2, 2, 256, 256, 64, 64, None, None, None, 0.125, 0.0, 1.0, None, None,
              null) == 1
    assert fm(fake, fake, fake, 1, 2, 2, 256, 256, 64, 64, None, None, fake, 0.125, 0.0, float("inf"), fake,
              fake, null) == 1
    fb = lib.splash_attention_bwd
    assert fb(None, None, None, None, None, None, 1, 2, 2, 256, 256, 64, 64, None, None, None, 0.125, 0.0,
              None, None, None, None, 0, null) == 1
    assert fb(fake, fake, fake, fake, fake, fake, 1, 2, 2, 256, 256, 64, 64, None, None, fake, -1.0, 0.0,
              fake, fake, fake, fake, 1 << 20, null) == 1
    n = ctypes.c_size_t(0)
    assert lib.splash_attention_bwd_workspace_size(2, 4, 1024, 128, ctypes.byref(n)) == 0
    assert n.value == 2 * 4 * 1024 * 128 * 4 + 2 * (2 * 4 * 1024 * 4)   # fp32 dq accumulator, D, LSE copy
    # a ragged Lq is padded to whole 128-row blocks per head
    assert lib.splash_attention_bwd_workspace_size(1, 2, 1000, 64, ctypes.byref(n)) == 0
    assert n.value == 2 * 1024 * 64 * 4 + 2 * (2 * 1024 * 4)
    assert lib.splash_attention_bwd_workspace_size(2, 4, 1024, 128, None) == 1
    assert lib.splash_mask_info_set_pattern_source(None, 0) == 1
    # counts / shape / to_host on a NULL handle
    assert lib.splash_mask_info_counts(None, None, None, None, None) == 1
    assert lib.splash_mask_info_shape(None, None, None, None, None, None) == 1
    lib.splash_mask_info_destroy(None)
    assert lib.splash_debug_wait_selftest(0, null) == 1
    assert lib.splash_debug_wait_selftest(3 * 10 ** 9, null) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, splash):
    monkeypatch.setattr(splash, "_lib", None)
    monkeypatch.setattr(splash, "LIB_PATH", "/nonexistent/libsplash.so")
    with pytest.raises(splash.SplashLibraryMissing):
        splash.lib()


def test_head_group_schedule(splash):
    """The forward's item order across heads (host logic, no device work)."""
    f = splash.lib().splash_schedule_head_group
    f.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
    f.restype = ctypes.c_int32
    MB = 1 << 20
    # wide-head causal MHA, 256-row q-blocks: 128 heads, 16 rows each, K / V 335 MB,
    # 152 CTAs -> 19 heads per group (two whole rounds)
    assert f(1, 16, 128, 128 * 4096 * 320 * 2, 152) == 19
    # dense causal GQA (33.5 MB of K / V) and anything that fits: no grouping
    assert f(1, 64, 16, 2 * 8 * 4096 * 256 * 2, 152) == 16
    assert f(1, 16, 128, 64 * MB, 152) == 128
    # windows / segment IDs: rows read short key ranges, no grouping
    assert f(0, 16, 128, 128 * 4096 * 320 * 2, 152) == 128
    assert f(1, 16, 1, 1 << 40, 152) == 1
    # invalid arguments
    assert f(1, 0, 8, MB, 152) == 0 and f(1, 16, 0, MB, 152) == 0 and f(1, 16, 8, MB, 0) == 0
    assert f(1, 16, 8, -1, 152) == 0
    # in general: between half the L2-sized bound and the bound, and no size
    # in that range leaves fewer items in a partial round
    import random
    rng = random.Random(7)
    for _ in range(200):
        npairs = rng.randint(2, 256)
        items = rng.randint(1, 200)
        grid = rng.choice([16, 132, 148, 152])
        kv = rng.randint(65 * MB, 4000 * MB)
        h = f(1, items, npairs, kv, grid)
        cap = max(1, npairs * (64 * MB) // kv)
        assert max(1, cap // 2) <= h <= cap
        assert all((items * h) % grid <= (items * x) % grid for x in range(max(1, cap // 2), cap + 1))


def test_shard_items_tile_the_groups(splash):
    for B, Hkv in ((1, 1), (2, 8), (1, 7), (3, 5), (5, 3)):
        n = B * Hkv
        for world in (1, 2, 3, 4, 8, 9):
            ranges = [splash.shard_items(B, Hkv, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            assert all(ranges[r][1] == ranges[r + 1][0] for r in range(world - 1))
            sizes = [e - b for b, e in ranges]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0
    lib = splash.lib()
    b, e = ctypes.c_int64(), ctypes.c_int64()
    for args in ((0, 1, 1, 0), (1, 0, 1, 0), (1, 1, 0, 0), (1, 1, 2, 2), (1, 1, 2, -1)):
        assert lib.splash_shard_items(*args, ctypes.byref(b), ctypes.byref(e)) == 1
    assert lib.splash_shard_items(1, 1, 1, 0, None, ctypes.byref(e)) == 1
