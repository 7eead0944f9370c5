"""The C-ABI library without a GPU: it builds, loads, exports every entry point
include/cpa.h declares, and rejects bad arguments on the host (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_prefill_attention_rope_gb300.build import build
    build()
    import chunked_prefill_attention_rope_gb300 as cpa
    return cpa, cpa.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "cpa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    _, so = lib
    names = declared_functions()
    assert len(names) == 13, names
    for name in names:
        assert hasattr(so, name), name


def test_checked_build_exports_the_same_symbols_and_its_hook(lib):
    """libcpa_checked.so (bounds checks and test hooks) exports every cpa.h
    entry point and cpa_test_drop_tile (include/cpa_test.h); the library
    itself has no test hook."""
    cpa, so = lib
    checked = cpa.load_library("checked")
    for name in declared_functions():
        assert hasattr(checked, name), name
    assert hasattr(checked, "cpa_test_drop_tile")
    assert not hasattr(so, "cpa_test_drop_tile")
    hdr = open(os.path.join(ROOT, "include", "cpa_test.h")).read()
    assert re.findall(r"\b(cpa_[a-z_]+)\s*\(", re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)) == ["cpa_test_drop_tile"]


def test_status_strings_and_version(lib):
    _, so = lib
    assert so.cpa_status_str(0) == b"ok"
    assert b"W <= C + S" in so.cpa_status_str(5)
    assert so.cpa_version().startswith(b"cpa")


def test_workspace_sizes(lib):
    cpa, so = lib
    # bad shapes -> 0; a decode-like step needs split-KV partials
    assert so.cpa_attn_workspace_size(1, 3, 2, 128, 1, 10) == 0
    assert so.cpa_attn_workspace_size(1, 4, 1, 96, 1, 10) == 0
    assert so.cpa_attn_workspace_size(64, 32, 8, 128, 1, 32768) > 0
    # an explicit mask on the two-tile path: room for a bit per mask entry on
    # top (16 bytes per row and 128-key tile); other paths need nothing more
    B, Hq, Hkv, D, C, P = 16, 32, 8, 128, 128, 4096
    plain = so.cpa_attn_workspace_size(B, Hq, Hkv, D, C, P)
    masked = so.cpa_attn_workspace_size_mask(B, Hq, Hkv, D, C, P)
    tiles = (C + 127) // 128 + (P + 127) // 128
    assert masked - plain >= B * Hq * C * tiles * 16
    assert masked - plain < B * Hq * C * tiles * 16 + 256
    assert so.cpa_attn_workspace_size_mask(1, 4, 1, 256, 64, 800) == so.cpa_attn_workspace_size(1, 4, 1, 256, 64, 800)
    assert so.cpa_attn_workspace_size_mask(1, 3, 2, 128, 1, 10) == 0


def _args(cpa, **kw):
    a = cpa._AttnArgs()
    a.B, a.Hq, a.Hkv, a.D, a.C, a.P = 1, 4, 1, 64, 16, 48
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_host_validation_returns_status_without_launch(lib):
    cpa, so = lib
    call = lambda a: so.cpa_chunk_prefill_attn(ctypes.byref(a), None)
    assert call(_args(cpa)) == 1                         # NULL pointers
    fake = 0x10000                                       # never dereferenced: validation fails first
    cache = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 64, fake, 64, 0, 0, 0)
    full = dict(q=fake, k_new=fake, v_new=fake, cos=fake, sin=fake, out=fake, err=fake,
                cache=ctypes.pointer(cache), past_len=fake, n_real=fake)
    assert call(_args(cpa, D=96, **full)) == 4           # unsupported head dim
    assert call(_args(cpa, Hq=3, Hkv=2, **full)) == 2    # Hq not a multiple of Hkv
    assert call(_args(cpa, P=65, **full)) == 2           # span beyond capacity
    assert call(_args(cpa, **dict(full, q=fake + 2))) == 3  # misaligned
    bad = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 68, fake, 64, 0, 0, 0)
    assert call(_args(cpa, **dict(full, cache=ctypes.pointer(bad)))) == 3  # stride not a multiple of 8
    assert so.cpa_decode_step(ctypes.byref(_args(cpa, **full)), None) == 2  # decode needs C == 1
    sl = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 64, fake, 64, 1, 32, 4)
    # an implicit mask over a sliding cache with sinks is accepted: validation
    # stops at the missing workspace, before any launch
    assert call(_args(cpa, **dict(full, cache=ctypes.pointer(sl)))) == 6
    # the fused attention + append takes global caches only, and needs n_rows
    fused = lambda a, n: so.cpa_chunk_prefill_attn_append(ctypes.byref(a), n, None)
    assert fused(_args(cpa, **dict(full, cache=ctypes.pointer(sl))), fake) == 4
    assert fused(_args(cpa, **full), None) == 1
    assert fused(_args(cpa, **full), fake + 4) == 3


def test_sliding_guards(lib):
    cpa, so = lib
    fake = 0x10000
    sl = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 64, fake, 64, 1, 24, 8)
    # W = 24 <= C + S = 16 + 8
    assert so.cpa_kv_snapshot_padded_append(ctypes.byref(sl), fake, 1, 1, 64, 16, fake, 1 << 30, fake, None) == 5
    assert so.cpa_kv_rollback_padded_append(ctypes.byref(sl), 1, 1, 64, 16, fake, 1 << 30, fake, None) == 5
    glob = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 64, fake, 64, 0, 0, 0)
    assert so.cpa_kv_snapshot_padded_append(ctypes.byref(glob), fake, 1, 1, 64, 16, fake, 1 << 30, fake, None) == 4
    ok = cpa._Cache(fake, fake, 64 * 64, 64 * 64, 64, fake, 64, 1, 40, 0)
    need = so.cpa_cache_scratch_size(ctypes.byref(ok), 1, 1, 64, 16)
    assert need > 0
    assert so.cpa_kv_snapshot_padded_append(ctypes.byref(ok), fake, 1, 1, 64, 16, fake, need - 1, fake, None) == 6
    assert so.cpa_cache_scratch_size(ctypes.byref(glob), 1, 1, 64, 16) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import chunked_prefill_attention_rope_gb300 as cpa
    monkeypatch.setattr(cpa, "_LIBS", {})
    monkeypatch.setattr(cpa, "lib_path", lambda variant=None: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        cpa.load_library()
    with pytest.raises(RuntimeError):
        cpa.load_library("checked")


def test_tail_plan_policy(lib):
    """cpa_tail_plan: scalar below the crossover, padded to the smallest
    bucket at or above it, the sink-aware window guard ("Pad the
    chunked-prefill tail for sliding-window models", Fix and review), and the
    kill switch."""
    cpa, _ = lib
    S, P = cpa.TAIL_SCALAR, cpa.TAIL_PADDED
    B4 = [16, 32, 64, 128]
    # the pages' M4 Pro policy: tails <= 8 stay scalar, padding from 9 up, one 128-row bucket
    assert cpa.tail_plan(8, 128, 512, 0, crossover=9) == (S, 8)
    assert cpa.tail_plan(9, 128, 512, 0, crossover=9) == (P, 128)
    assert cpa.tail_plan(127, 128, 512, 0, crossover=9) == (P, 128)
    # buckets: the smallest one that holds the tail
    assert cpa.tail_plan(9, 128, 512, 0, B4, crossover=9) == (P, 16)
    assert cpa.tail_plan(16, 128, 512, 0, B4, crossover=9) == (P, 16)
    assert cpa.tail_plan(17, 128, 512, 0, B4, crossover=9) == (P, 32)
    assert cpa.tail_plan(100, 128, 512, 0, B4, crossover=9) == (P, 128)
    # library default crossover
    assert cpa.tail_plan(1, 128, 512, 0, B4) == (S, 1)
    assert cpa.tail_plan(2, 128, 512, 0, B4) == (P, 16)
    # sink-aware guard: W <= c_pad + S is never snapshotted; a larger bucket
    # cannot help, so the tail stays scalar (or a forced pad is refused)
    assert cpa.tail_plan(20, 32, 40, 0, [16, 32], crossover=9) == (P, 32)
    assert cpa.tail_plan(20, 32, 40, 8, [16, 32], crossover=9) == (S, 20)
    assert cpa.tail_plan(12, 32, 40, 8, [16, 32], crossover=9) == (P, 16)
    with pytest.raises(cpa.CpaError) as e:
        cpa.tail_plan(20, 32, 40, 8, [16, 32], force=cpa.TAIL_FORCE_PADDED)
    assert e.value.status == 5
    # global caches have no window guard
    assert cpa.tail_plan(20, 32, 0, 0, [16, 32], crossover=9) == (P, 32)
    # kill switch and forced padding
    assert cpa.tail_plan(127, 128, 512, 0, B4, force=cpa.TAIL_FORCE_SCALAR) == (S, 127)
    assert cpa.tail_plan(1, 128, 512, 0, B4, force=cpa.TAIL_FORCE_PADDED) == (P, 16)
    # bad arguments
    for bad in (dict(t=0, C=128), dict(t=129, C=128), dict(t=4, C=128, buckets=[32, 16]),
                dict(t=4, C=128, buckets=[16, 256]), dict(t=4, C=128, window=-1), dict(t=4, C=128, force=3)):
        with pytest.raises(cpa.CpaError) as e:
            cpa.tail_plan(**bad)
        assert e.value.status == 2, bad
