"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol that include/sattn.h declares; invalid arguments are rejected on the
host before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(sattn_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from windowed_attention_sinks_gb300 import build

    build.build()
    import windowed_attention_sinks_gb300 as sa

    return sa.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sattn_window_fwd", "sattn_sparse_fwd", "sattn_merge_lse",
              "sattn_block_sparse_fwd", "sattn_sparse_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in sorted(_declared()):
        assert hasattr(lib, n), "missing export %s" % n


def test_status_strings(lib):
    for code in range(6):
        assert lib.sattn_status_str(code)
    assert lib.sattn_version() >= 100


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # H % Hkv != 0
    rc = lib.sattn_window_fwd(fake, fake, fake, fake, None, fake, 1, 10, 10, 6, 4, 128, 8, 8, 0,
                              None, 0, 0.1, 1, None)
    assert rc == 1
    # d not in {64, 128}
    rc = lib.sattn_window_fwd(fake, fake, fake, fake, None, fake, 1, 10, 10, 8, 4, 96, 8, 8, 0,
                              None, 0, 0.1, 1, None)
    assert rc == 1
    # sink mode without sinks
    rc = lib.sattn_window_fwd(fake, fake, fake, fake, None, fake, 1, 10, 10, 8, 4, 128, 8, 8, 0,
                              None, 1, 0.1, 1, None)
    assert rc == 1
    # NaN scale
    rc = lib.sattn_window_fwd(fake, fake, fake, fake, None, fake, 1, 10, 10, 8, 4, 128, 8, 8, 0,
                              None, 0, float("nan"), 1, None)
    assert rc == 1
    # NULL q
    rc = lib.sattn_window_fwd(None, fake, fake, fake, None, fake, 1, 10, 10, 8, 4, 128, 8, 8, 0,
                              None, 0, 0.1, 1, None)
    assert rc == 1
    # empty work is a no-op
    rc = lib.sattn_window_fwd(None, None, None, None, None, None, 0, 0, 0, 8, 4, 128, 8, 8, 0,
                              None, 0, 0.1, 1, None)
    assert rc == 0
    # sparse: negative K, misaligned workspace, bf16 with d=64
    rc = lib.sattn_sparse_fwd(fake, fake, fake, None, 0, 0.1, fake, None, 1, 1, 32, 128, 10, -1,
                              None, 0, 1, None)
    assert rc == 1
    rc = lib.sattn_sparse_fwd(fake, fake, fake, None, 0, 0.1, fake, None, 1, 1, 32, 128, 10, 5,
                              P(0x1004), 4096, 1, None)
    assert rc == 1
    rc = lib.sattn_sparse_fwd(fake, fake, fake, None, 0, 0.1, fake, None, 1, 1, 32, 64, 10, 5,
                              None, 0, 1, None)
    assert rc == 2
    rc = lib.sattn_sparse_fwd(None, None, None, None, 0, 0.1, None, None, 0, 5, 32, 128, 10, 5,
                              None, 0, 1, None)
    assert rc == 0
    # block sparse: kv range outside the context
    rc = lib.sattn_block_sparse_fwd(fake, fake, fake, fake, 4, 100, 8, 4, 128, 0, 0, 101, 1, 0.1,
                                    fake, fake, 1, None)
    assert rc == 1
    # merge: bad d
    # index lists: win < 1, negative ratio
    assert lib.sattn_build_topk_idxs(fake, fake, 1, 4, 16, 0, 4, None) == 1
    assert lib.sattn_build_topk_idxs(fake, fake, 1, 4, 16, 8, -1, None) == 1
    assert lib.sattn_build_topk_idxs(None, None, 0, 4, 16, 8, 4, None) == 0  # empty: no work
    # ring write: N < win, row bytes not a multiple of 16, misaligned pointer
    assert lib.sattn_kv_ring_write(fake, fake, fake, 1, 4, 4, 128, 8, 1, None) == 1
    assert lib.sattn_kv_ring_write(fake, fake, fake, 1, 4, 16, 3, 8, 1, None) == 1
    assert lib.sattn_kv_ring_write(ctypes.c_void_p(fake.value + 4), fake, fake, 1, 4, 16, 128, 8,
                                   1, None) == 1
    rc = lib.sattn_merge_lse(fake, fake, 2, 10, 0, 8, None, fake, None, 0, None)
    assert rc == 1
    # compressor: d not a multiple of 4, ratio 0, bad overlap flag, out stride
    # too small, misaligned pointer; fewer tokens than a window is no work
    i64 = ctypes.c_int64
    assert lib.sattn_compress_kv(fake, fake, fake, fake, i64(1000), 2, 64, 6, 4, 1, 0, 0,
                                 None) == 1
    assert lib.sattn_compress_kv(fake, fake, fake, fake, i64(1000), 2, 64, 8, 0, 1, 0, 0,
                                 None) == 1
    assert lib.sattn_compress_kv(fake, fake, fake, fake, i64(1000), 2, 64, 8, 4, 2, 0, 0,
                                 None) == 1
    assert lib.sattn_compress_kv(fake, fake, fake, fake, i64(124), 2, 64, 8, 4, 1, 0, 0,
                                 None) == 1
    assert lib.sattn_compress_kv(fake, ctypes.c_void_p(fake.value + 8), fake, fake, i64(128), 2,
                                 64, 8, 4, 1, 0, 0, None) == 1
    assert lib.sattn_compress_kv(None, None, None, None, i64(0), 2, 3, 8, 4, 1, 0, 0,
                                 None) == 0
    # FP8 layout: rd > d, d not a multiple of 4, misaligned output; gathered
    # attention over it: unsupported shape, missing scale array
    assert lib.sattn_quantize_kv_fp8(fake, fake, fake, fake, i64(4), 128, 130, 1, None) == 1
    assert lib.sattn_quantize_kv_fp8(fake, fake, fake, fake, i64(4), 126, 62, 1, None) == 1
    assert lib.sattn_quantize_kv_fp8(fake, ctypes.c_void_p(fake.value + 4), fake, fake, i64(4),
                                     128, 64, 1, None) == 1
    assert lib.sattn_quantize_kv_fp8(None, None, None, None, i64(0), 128, 64, 1, None) == 0
    f32 = ctypes.c_float
    assert lib.sattn_sparse_fp8_fwd(fake, fake, fake, fake, fake, None, 0, f32(0.1), fake, None,
                                    1, 1, 16, 128, 64, 8, 8, None, 0, None) == 2
    assert lib.sattn_sparse_fp8_fwd(fake, fake, fake, None, fake, None, 0, f32(0.1), fake, None,
                                    1, 1, 32, 128, 64, 8, 8, None, 0, None) == 1
    # block selection: chunk not on a block boundary, H % Hkv, d != 128,
    # threshold out of range
    assert lib.sattn_xattn_partial_stats(fake, fake, 4, 512, 4, 2, 128, 0, 64, 512, 1, f32(0.1),
                                         fake, fake, None) == 1
    assert lib.sattn_xattn_partial_stats(fake, fake, 4, 512, 4, 3, 128, 0, 0, 512, 1, f32(0.1),
                                         fake, fake, None) == 1
    assert lib.sattn_xattn_partial_stats(fake, fake, 4, 512, 4, 2, 64, 0, 0, 512, 1, f32(0.1),
                                         fake, fake, None) == 2
    assert lib.sattn_xattn_block_sum(fake, fake, fake, fake, 4, 512, 4, 2, 128, 0, 0, 500, 1,
                                     f32(0.1), fake, None) == 1
    assert lib.sattn_xattn_find_blocks(fake, 2, 2, 4, f32(1.5), fake, None) == 1
    assert lib.sattn_xattn_find_blocks(fake, 2, 2, 5000, f32(0.9), fake, None) == 1
    assert lib.sattn_xattn_merge_stats(None, None, 0, 0, None, None, None) == 0
    # all chunks at once: chunk <= 0, range past Nctx, H % Hkv; an empty
    # range or no rows is no work
    assert lib.sattn_block_sparse_chunks_fwd(fake, fake, fake, fake, 128, 1024, 4, 2, 128, 0, 0,
                                             1024, 0, 1, f32(0.1), fake, fake, 1, None) == 1
    assert lib.sattn_block_sparse_chunks_fwd(fake, fake, fake, fake, 128, 1024, 4, 2, 128, 0, 0,
                                             2048, 256, 1, f32(0.1), fake, fake, 1, None) == 1
    assert lib.sattn_block_sparse_chunks_fwd(fake, fake, fake, fake, 128, 1024, 4, 3, 128, 0, 0,
                                             1024, 256, 1, f32(0.1), fake, fake, 1, None) == 1
    assert lib.sattn_block_sparse_chunks_fwd(None, None, None, None, 128, 1024, 4, 2, 128, 0, 512,
                                             512, 256, 1, f32(0.1), None, None, 1, None) == 0
    assert lib.sattn_block_sparse_chunks_fwd(None, None, None, None, 0, 1024, 4, 2, 128, 0, 0,
                                             1024, 256, 1, f32(0.1), None, None, 1, None) == 0
    # the one-call selection: chunk not a multiple of 128 or 0, threshold out
    # of range, workspace too small or misaligned, too many key blocks, more
    # heads than a grid dimension holds; no rows is no work
    ws = lib.sattn_xattn_select_workspace_bytes(256, 4, 1024, 256)

    def sel(M=256, Nctx=1024, H=4, chunk=256, thr=0.9, w=fake, nb=ws):
        return lib.sattn_xattn_select_blocks(fake, fake, M, Nctx, H, 2, 128, 0, 1, f32(0.1), chunk,
                                             f32(thr), w, nb, fake, fake, None)
    assert sel(chunk=200) == 1
    assert sel(chunk=0) == 1
    assert sel(thr=1.5) == 1
    assert sel(nb=ws - 4) == 1
    assert sel(w=ctypes.c_void_p(fake.value + 8)) == 1
    assert sel(Nctx=4097 * 128, chunk=128 * 4097) == 1
    assert sel(H=65536 * 2) == 1
    assert sel(M=0, w=None, nb=0) == 0


def test_select_workspace_bytes(lib):
    # per-chunk (m, l) and the merged (m, l), float32 [2 C + 2, M, H]
    assert lib.sattn_xattn_select_workspace_bytes(256, 4, 1024, 256) == (2 * 4 + 2) * 256 * 4 * 4
    assert lib.sattn_xattn_select_workspace_bytes(100, 3, 1000, 384) == (2 * 3 + 2) * 100 * 3 * 4
    assert lib.sattn_xattn_select_workspace_bytes(0, 4, 1024, 256) == 0
    assert lib.sattn_xattn_select_workspace_bytes(256, 4, 1024, 0) == 0


def test_workspace_size_monotone(lib):
    small = lib.sattn_sparse_workspace_bytes(1, 1, 32, 128, 640)
    big = lib.sattn_sparse_workspace_bytes(64, 1, 32, 128, 640)
    assert big >= small >= 0
    assert lib.sattn_sparse_workspace_bytes(0, 1, 32, 128, 640) == 0


def test_workspace_bytes_for_huge_batches(lib):
    # B * M beyond 32 bits needs no split (and must not overflow or divide by zero)
    assert lib.sattn_sparse_workspace_bytes(65536, 65536, 32, 128, 640) == 0
    assert lib.sattn_sparse_workspace_bytes(2 ** 31 - 1, 2, 32, 128, 640) == 0
    assert lib.sattn_sparse_workspace_bytes(2 ** 31 - 1, 2 ** 31 - 1, 32, 128, 640) == 0
