"""The C-ABI library builds, loads and exports every symbol include/kvr.h
declares; host-only calls behave (no GPU needed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
import workloads


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from prefix_reused_prefill_gb300 import kvr
    return kvr.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvr_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    from prefix_reused_prefill_gb300 import kvr
    assert sorted(kvr.EXPORTED) == names


def test_sizes_match_documented_layout(lib):
    from prefix_reused_prefill_gb300 import kvr
    shape = workloads.SHAPES["qwen7b"]
    cfg = kvr.config_for_shape(shape, 4, 16384, 256)
    per_slot = shape.n_layers * 2 * shape.n_kv_heads * 16384 * shape.head_dim * 2 + 16384 * 4
    assert lib.kvr_arena_bytes(ctypes.byref(cfg), 4) == 4 * per_slot
    assert lib.kvr_arena_bytes(ctypes.byref(cfg), 1) == per_slot
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) > 0


@pytest.mark.parametrize("field,value", [("capacity", 100), ("head_dim", 96), ("n_kv_heads", 3),
                                         ("n_slots", 17), ("max_rows", 0), ("weight_format", 7),
                                         ("vocab", -1), ("vocab", 262145)])
def test_invalid_configs_are_refused(lib, field, value):
    from prefix_reused_prefill_gb300 import kvr
    cfg = kvr.config_for_shape(workloads.SHAPES["qwen7b"], 4, 16384, 256)
    setattr(cfg, field, value)
    assert lib.kvr_arena_bytes(ctypes.byref(cfg), 1) == 0
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) == 0
    out = ctypes.c_void_p()
    assert lib.kvr_ctx_create(ctypes.byref(cfg), None, 0, None, 0, ctypes.byref(out)) == -1


def test_q4k_is_a_format(lib):
    from prefix_reused_prefill_gb300 import kvr
    cfg = kvr.config_for_shape(workloads.SHAPES["small_q4k"], 2, 256, 32)
    assert cfg.weight_format == 2 and lib.kvr_scratch_bytes(ctypes.byref(cfg)) > 0
    cfg.hidden = 640  # the input widths follow the int4 rule
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) == 0
    cfg = kvr.config_for_shape(workloads.SHAPES["small_q4k"], 2, 256, 32)
    cfg.weight_format = 3
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) == 0


def test_int4_width_rule(lib):
    from prefix_reused_prefill_gb300 import kvr
    cfg = kvr.config_for_shape(workloads.SHAPES["small"], 2, 256, 32)
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) > 0
    cfg.hidden = 640  # not a multiple of 256
    assert lib.kvr_scratch_bytes(ctypes.byref(cfg)) == 0


def test_output_head_scratch_grows_with_vocab(lib):
    """The scratch holds, per verify row and 128-row LM-head tile, one (value, index) pair,
    and the head GEMV's partial sums (three contributions per tile at most)."""
    from prefix_reused_prefill_gb300 import kvr
    shape = workloads.SHAPES["small"]
    base = lib.kvr_scratch_bytes(ctypes.byref(kvr.config_for_shape(shape, 2, 256, 32)))
    for vocab in (1000, 32000, 262144):
        cfg = kvr.config_for_shape(shape, 2, 256, 32, vocab=vocab)
        tiles = -(-vocab // 128)
        grow = lib.kvr_scratch_bytes(ctypes.byref(cfg)) - base
        assert grow >= 64 * tiles * 8 - 256   # the vocab-0 layout keeps one aligned block
        assert grow <= 64 * tiles * 8 + tiles * 3 * 32 * 128 * 4 + 4096


def _fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: offset basis 14695981039346656037, prime 1099511628211."""
    h = 14695981039346656037
    for byte in data:
        h = ((h ^ byte) * 1099511628211) % (1 << 64)
    return h


def test_fnv1a_reference_vectors():
    # the published FNV-1a 64-bit values of the empty string and of "a"
    assert _fnv1a64(b"") == 0xcbf29ce484222325
    assert _fnv1a64(b"a") == 0xaf63dc4c8601ec8c


def test_config_hash_is_fnv1a_of_the_kv_fields(lib):
    import struct
    from prefix_reused_prefill_gb300 import kvr
    cfg = kvr.config_for_shape(workloads.SHAPES["dense9b"], 4, 8192, 256)
    for tag in (0, 1, 0x0123456789abcdef):
        words = struct.pack("<8I", cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                            cfg.ffn, cfg.weight_format, cfg.attn_only)
        words += struct.pack("<2f", cfg.rope_theta, cfg.rms_eps) + struct.pack("<Q", tag)
        assert lib.kvr_config_hash(ctypes.byref(cfg), tag) == _fnv1a64(words)


def test_config_hash_sees_the_kv_fields_only(lib):
    from prefix_reused_prefill_gb300 import kvr
    base = kvr.config_for_shape(workloads.SHAPES["dense9b"], 4, 8192, 256)
    h0 = lib.kvr_config_hash(ctypes.byref(base), 7)
    assert lib.kvr_config_hash(ctypes.byref(base), 8) != h0
    for field, value in [("n_layers", 35), ("hidden", 4352), ("n_q_heads", 16), ("n_kv_heads", 4),
                         ("head_dim", 64), ("ffn", 12544), ("weight_format", 0), ("attn_only", 1),
                         ("rope_theta", 5e5), ("rms_eps", 1e-5)]:
        cfg = kvr.config_for_shape(workloads.SHAPES["dense9b"], 4, 8192, 256)
        setattr(cfg, field, value)
        assert lib.kvr_config_hash(ctypes.byref(cfg), 7) != h0, field
    for field, value in [("n_slots", 1), ("capacity", 16384), ("max_rows", 64), ("match_threshold", 0),
                         ("vocab", 32000)]:
        cfg = kvr.config_for_shape(workloads.SHAPES["dense9b"], 4, 8192, 256)
        setattr(cfg, field, value)
        assert lib.kvr_config_hash(ctypes.byref(cfg), 7) == h0, field


def test_null_context_calls_return_arg_errors(lib):
    n = ctypes.c_int()
    assert lib.kvr_slot_len(None, 0, ctypes.byref(n)) == -1
    assert lib.kvr_slot_truncate(None, 0, 0) == -1
    assert lib.kvr_ctx_destroy(None) == -1
    acc = ctypes.c_int()
    assert lib.kvr_verify_accept(None, 0, None, 1, None, None, None, None, None, ctypes.byref(acc), None) == -1
    assert lib.kvr_slot_spill_bytes(None, 0) == 0
    assert lib.kvr_slot_spill(None, 0, 0, None, 0, None) == -1
    assert lib.kvr_slot_restore(None, 0, 0, None, 0, None) == -1
    assert lib.kvr_last_error(None) == b"null context"


def test_binding_fails_loudly_without_library(tmp_path):
    from prefix_reused_prefill_gb300 import kvr
    saved = kvr._lib
    try:
        kvr._lib = None
        with pytest.raises(ImportError):
            kvr.load_library(str(tmp_path / "missing.so"))
    finally:
        kvr._lib = saved


def test_token_ids_marshal_to_int32_arrays():
    """The binding hands token ids to the C ABI as one int32 array: a list goes
    through a single array copy, an int32 numpy array is passed as it is, other
    integer arrays are converted, an empty list still gives a valid pointer, and
    ids outside int32 are refused rather than wrapped."""
    import numpy as np
    from prefix_reused_prefill_gb300.kvr import _i32
    a = _i32([5, 0, 151935, 2**31 - 1])
    assert isinstance(a, ctypes.Array) and ctypes.sizeof(a._type_) == 4
    assert list(a) == [5, 0, 151935, 2**31 - 1]
    assert list(_i32([np.int64(7), np.int32(3)])) == [7, 3]
    assert list(_i32([])) == [0]
    n32 = np.arange(10, 20, dtype=np.int32)
    b = _i32(n32)
    assert list(b) == list(range(10, 20))
    assert ctypes.addressof(b) == n32.ctypes.data          # no copy
    assert list(_i32(np.array([[1, 2], [3, 4]], dtype=np.int64))) == [1, 2, 3, 4]
    ro = np.arange(3, dtype=np.int32)
    ro.flags.writeable = False
    assert list(_i32(ro)) == [0, 1, 2]
    with pytest.raises(OverflowError):
        _i32([2**31])
