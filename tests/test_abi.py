"""The C ABI library: it loads, exports every declared symbol, and its
host-side logic (validation, sizes) answers without touching a GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

from helpers import ROOT, ensure_library


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "fm.h")).read()
    return sorted(set(re.findall(r"FM_API[^;(]*?\b(fm_\w+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("fm_rope_qk_varlen", "fm_mask_block_minmax", "fm_attn_fwd_varlen"):
        assert n in names


def test_every_declared_symbol_is_exported(fm):
    lib = ctypes.CDLL(fm.library_path())
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(fm.EXPORTED_SYMBOLS) == _declared()


def test_status_strings_and_version(fm):
    assert fm.version() >= 100
    assert fm.status_string(0) == "FM_OK"
    assert fm.status_string(6) == "FM_ERR_TIMEOUT"
    assert fm.status_string(99) == "FM_ERR_UNKNOWN"


def test_kv_tile_bound_and_slot_layout(fm):
    assert fm.num_kv_tiles_bound(256, 3, 64) == 4 + 3
    assert fm.num_kv_tiles_bound(-1, 3, 64) == -1
    rng = np.random.default_rng(0)
    for _ in range(50):
        lens = rng.integers(0, 700, size=rng.integers(1, 12))
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        T = int(cu[-1])
        for bn in (64, 128):
            bound = fm.num_kv_tiles_bound(T, len(lens), bn)
            used = set()
            for s, n in enumerate(lens):
                for j in range(-(-int(n) // bn)):
                    slot = int(cu[s]) // bn + s + j
                    assert 0 <= slot < bound and slot not in used
                    used.add(slot)


def test_workspace_size(fm):
    a = fm.attn_fwd_workspace_size(8192, 30, 32, 128)
    b = fm.attn_fwd_workspace_size(8192, 30, 32, 64)
    assert a > 0 and b > a and a % 256 == 0
    assert fm.attn_fwd_workspace_size(10, 1, 1, 96) == 0


def _raw(fm):
    return fm._lib()


def test_validation_rejects_before_any_launch(fm):
    lib = _raw(fm)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    # unsupported head_dim
    assert lib.fm_rope_qk_varlen(fake, fake, 16, 1, 1, 96, 96, 96, fake, 1, 1e4, 0, 0, None) == 2
    # null q
    assert lib.fm_rope_qk_varlen(None, fake, 16, 1, 1, 64, 64, 64, fake, 1, 1e4, 0, 0, None) == 1
    # misaligned q
    assert lib.fm_rope_qk_varlen(ctypes.c_void_p(0x10002), fake, 16, 1, 1, 64, 64, 64, fake, 1,
                                 1e4, 0, 0, None) == 3
    # bad theta, unknown flag
    assert lib.fm_rope_qk_varlen(fake, fake, 16, 1, 1, 64, 64, 64, fake, 1, -1.0, 0, 0, None) == 1
    assert lib.fm_rope_qk_varlen(fake, fake, 16, 1, 1, 64, 64, 64, fake, 1, 1e4, 0, 8, None) == 1
    # minmax: capacity too small, bad block size
    assert lib.fm_mask_block_minmax(fake, 1, 256, fake, 3, 64, fake, 10, None) == 4
    assert lib.fm_mask_block_minmax(fake, 1, 256, fake, 3, 96, fake, 10 ** 6, None) == 2
    # attention: GQA ratio, mask heads, block sizes, workspace, alignment
    def attn(hq=4, hkv=2, d=128, sri=None, hm=0, mm=None, bm=128, bn=128, ws_bytes=1 << 20,
             ws=fake, out=fake):
        return lib.fm_attn_fwd_varlen(fake, fake, fake, 256, hq, hkv, d, fake, 2, sri, hm, mm, 1,
                                      0.0, bm, bn, out, fake, None, ws, ws_bytes, 0, None)
    assert attn(hq=3, hkv=2) == 1
    assert attn(sri=fake, hm=2, mm=fake) == 1
    assert attn(sri=fake, hm=1, mm=None) == 1
    assert attn(sri=None, mm=fake) == 1
    assert attn(d=96) == 2
    assert attn(bm=32) == 2
    assert attn(ws_bytes=16) == 4
    assert attn(ws=ctypes.c_void_p(0x10010)) == 3
    assert attn(out=ctypes.c_void_p(0x10008)) == 3
    # fused RoPE attention: theta, k, q_rot alignment, then the same checks
    def attn_rope(theta=1e4, k=fake, q_rot=None, hq=4, hkv=2):
        return lib.fm_attn_fwd_varlen_rope(fake, k, fake, 256, hq, hkv, 128, fake, 2, theta,
                                           None, 0, None, 1, 0.0, 128, 128, fake, fake, q_rot,
                                           None, fake, 1 << 20, 0, None)
    assert attn_rope(theta=0.0) == 1
    assert attn_rope(theta=-5.0) == 1
    assert attn_rope(theta=float("inf")) == 1
    assert attn_rope(k=None) == 1
    assert attn_rope(q_rot=ctypes.c_void_p(0x10008)) == 3
    assert attn_rope(hq=3) == 1
    # the scheduler alone: the same sample, mask, tile and workspace rules
    def plan(cu=fake, hq=4, hkv=2, sri=None, hm=0, mm=None, bm=128, bn=128, ws=fake,
             ws_bytes=1 << 20, T=256):
        return lib.fm_attn_fwd_plan(T, hq, hkv, cu, 2, sri, hm, mm, 1, bm, bn, ws, ws_bytes, None)
    assert plan(cu=None) == 1
    assert plan(ws=None) == 1
    assert plan(T=-1) == 1
    assert plan(hq=0) == 1
    assert plan(hq=4, hkv=3) == 1
    assert plan(hkv=0) == 1
    assert plan(sri=fake, hm=3, mm=fake) == 1
    assert plan(sri=fake, hm=1, mm=None) == 1
    assert plan(bm=96) == 2
    assert plan(bn=32) == 2
    assert plan(ws=ctypes.c_void_p(0x10010)) == 3
    assert plan(ws_bytes=16) == 4
    assert plan(T=0) == 0  # nothing to schedule: no launch
    # flags: unknown bits are refused; the allocation-free call never reuses a plan
    assert lib.fm_attn_fwd_varlen(fake, fake, fake, 256, 4, 2, 128, fake, 2, None, 0, None, 1,
                                  0.0, 128, 128, fake, fake, None, fake, 1 << 20, 4, None) == 1
    assert lib.fm_attn_fwd_varlen_noalloc(fake, fake, fake, 256, 4, 2, 128, fake, 2, None, 0, None,
                                          1, 0.0, 128, 128, fake, fake, None,
                                          fm.FM_FLAG_REUSE_PLAN, None) == 1
    assert lib.fm_debug_bounded_wait(fake, 0, None) == 1


def test_index_width_switches_at_2_pow_31(fm):
    """Int64 indexing only where an element offset can reach 2^31 (host-only:
    the same function the calls use to pick their instantiation)."""
    lim = 1 << 31
    # attention: T * Hq * D or T * Hkv * D reaching 2^31
    assert fm.attn_index_bits(lim // (32 * 128) - 1, 32, 8, 128) == 32
    assert fm.attn_index_bits(lim // (32 * 128), 32, 8, 128) == 64
    assert fm.attn_index_bits(lim // (8 * 128), 1, 8, 128) == 64   # via the key/value heads
    assert fm.attn_index_bits(131072, 32, 8, 128) == 32            # 2^29: only forced
    assert fm.attn_index_bits(131072, 32, 8, 128, force_int64=True) == 64
    assert fm.attn_index_bits(-1, 32, 8, 128) == -1
    # RoPE: T * token stride of q or k, or T * D / 16 threads
    assert fm.rope_index_bits(8192, 8, 128, 32 * 128, 8 * 128) == 32
    assert fm.rope_index_bits(lim // 4096, 8, 128, 4096, 1024) == 64
    assert fm.rope_index_bits(lim // 4096 - 1, 8, 128, 4096, 1024) == 32
    assert fm.rope_index_bits(lim // 1024, 8, 128, 128, 1024) == 64   # k stride
    assert fm.rope_index_bits(lim // 1024, 0, 128, 128, 1 << 40) == 32  # no k heads
    assert fm.rope_index_bits(8192, 8, 128, 4096, 1024, force_int64=True) == 64


def test_header_compiles_as_c_and_links(fm, tmp_path):
    """A plain C99 program builds against include/fm.h, links libfm.so and
    gets the expected answers from the calls that need no GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(fm.library_path())
    exe = str(tmp_path / "abi_from_c")
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                    "-o", exe, "-L", lib_dir, "-lfm", "-Wl,-rpath," + lib_dir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok FM_ERR_WORKSPACE"
