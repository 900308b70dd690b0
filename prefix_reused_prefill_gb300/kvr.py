"""ctypes binding of libkvr (include/kvr.h): argument marshalling only.

Torch is used for device memory (the KV arena, scratch, inputs, outputs) and
streams; every step of the suffix prefill runs in libkvr's kernels.  If the
library is not built this module raises on first use -- there is no fallback.
"""
from __future__ import annotations

import array
import ctypes
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvr.so")

KVR_OK = 0
ERRORS = {-1: "KVR_ERR_ARG", -2: "KVR_ERR_CAPACITY", -3: "KVR_ERR_CUDA", -4: "KVR_ERR_TIMEOUT",
          -5: "KVR_ERR_FAULT", -6: "KVR_ERR_UNSUPPORTED", -7: "KVR_ERR_MISMATCH"}
WEIGHTS_BF16, WEIGHTS_INT4_G32, WEIGHTS_Q4K = 0, 1, 2
_FORMATS = {"bf16": WEIGHTS_BF16, "int4": WEIGHTS_INT4_G32, "q4k": WEIGHTS_Q4K}
MAX_SLOTS, MAX_BRANCHES = 16, 16

EXPORTED = ["kvr_arena_bytes", "kvr_scratch_bytes", "kvr_ctx_create", "kvr_ctx_info",
            "kvr_ctx_destroy", "kvr_slot_match", "kvr_slot_truncate", "kvr_slot_len",
            "kvr_slot_tokens", "kvr_slot_assign", "kvr_slot_kv", "kvr_prefill_suffix", "kvr_verify",
            "kvr_prefill_branches", "kvr_sync_status", "kvr_profile_enable", "kvr_profile_read",
            "kvr_profile_launches",
            "kvr_last_error", "kvr_slot_match_static", "kvr_trace_set", "kvr_verify_accept",
            "kvr_config_hash", "kvr_slot_spill_bytes", "kvr_slot_spill", "kvr_slot_restore",
            "kvr_prefill_batch", "kvr_selftest_wait", "kvr_verify_accept_batch"]


class KvrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class KvrConfig(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int), ("capacity", ctypes.c_int), ("n_layers", ctypes.c_int),
                ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("weight_format", ctypes.c_int),
                ("attn_only", ctypes.c_int), ("match_threshold", ctypes.c_int),
                ("max_rows", ctypes.c_int), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("vocab", ctypes.c_int)]


_W_FIELDS = ["wq", "wk", "wv", "wo", "wg", "wu", "wd", "sq", "sk", "sv", "so", "sg", "su", "sd",
             "norm_attn", "norm_ffn"]


class KvrLayerWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in _W_FIELDS]


class KvrHeadWeights(ctypes.Structure):
    _fields_ = [("norm", ctypes.c_void_p), ("w", ctypes.c_void_p), ("s", ctypes.c_void_p),
                ("vocab", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH):
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libkvr.so not built at {path}: run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, Z, V = ctypes.POINTER, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    i32p = P(ctypes.c_int32)
    sig = {
        "kvr_arena_bytes": (Z, [P(KvrConfig), I]),
        "kvr_scratch_bytes": (Z, [P(KvrConfig)]),
        "kvr_ctx_create": (I, [P(KvrConfig), V, Z, V, Z, P(V)]),
        "kvr_ctx_info": (I, [V, P(I), P(I), P(I)]),
        "kvr_ctx_destroy": (I, [V]),
        "kvr_slot_match": (I, [V, i32p, I, P(I), P(I), V]),
        "kvr_slot_truncate": (I, [V, I, I]),
        "kvr_slot_len": (I, [V, I, P(I)]),
        "kvr_slot_tokens": (I, [V, I, i32p, I]),
        "kvr_slot_assign": (I, [V, I, i32p, I, V]),
        "kvr_slot_kv": (I, [V, I, I, P(V), P(V)]),
        "kvr_prefill_suffix": (I, [V, I, i32p, I, V, P(KvrLayerWeights), V, V]),
        "kvr_verify": (I, [V, I, i32p, I, V, P(KvrLayerWeights), V, V]),
        "kvr_verify_accept": (I, [V, I, i32p, I, V, P(KvrLayerWeights), P(KvrHeadWeights), V, i32p,
                                  P(I), V]),
        "kvr_prefill_branches": (I, [V, I, I, P(I), i32p, V, P(KvrLayerWeights), V, V]),
        "kvr_prefill_batch": (I, [V, I, P(I), P(I), i32p, V, P(KvrLayerWeights), V, V]),
        "kvr_sync_status": (I, [V, V]),
        "kvr_profile_enable": (I, [V, I]),
        "kvr_profile_read": (I, [V, P(ctypes.c_float), P(I)]),
        "kvr_profile_launches": (I, [V, P(I), P(ctypes.c_float), I, P(I)]),
        "kvr_last_error": (ctypes.c_char_p, [V]),
        "kvr_slot_match_static": (I, [V, i32p, I, P(I), P(I), V]),
        "kvr_trace_set": (I, [V, V, Z]),
        "kvr_selftest_wait": (I, [V, V]),
        "kvr_verify_accept_batch": (I, [V, I, P(I), P(I), i32p, V, P(KvrLayerWeights), P(KvrHeadWeights), V,
                                        i32p, P(I), V]),
        "kvr_config_hash": (ctypes.c_uint64, [P(KvrConfig), ctypes.c_uint64]),
        "kvr_slot_spill_bytes": (Z, [V, I]),
        "kvr_slot_spill": (I, [V, I, ctypes.c_uint64, V, Z, V]),
        "kvr_slot_restore": (I, [V, I, ctypes.c_uint64, V, Z, V]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def config_for_shape(shape, n_slots: int, capacity: int, max_rows: int,
                     match_threshold: bool = True, n_layers: Optional[int] = None,
                     vocab: int = 0) -> KvrConfig:
    return KvrConfig(n_slots, capacity, shape.n_layers if n_layers is None else n_layers,
                     shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                     shape.ffn, _FORMATS[shape.weight_format],
                     1 if shape.attn_only else 0, 1 if match_threshold else 0, max_rows,
                     shape.rope_theta, shape.rms_eps, vocab)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def layer_weight_structs(layers: Sequence[Dict[str, object]]):
    """workloads-style layer dicts -> (ctypes array, tensors kept alive)."""
    arr = (KvrLayerWeights * len(layers))()
    keep: List[torch.Tensor] = []
    for i, lw in enumerate(layers):
        for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            v = lw.get(name)
            if v is None:
                continue
            if hasattr(v, "packed"):
                setattr(arr[i], name, _ptr(v.packed))
                setattr(arr[i], "s" + name[1], _ptr(v.scales))
                keep += [v.packed, v.scales]
            else:
                setattr(arr[i], name, _ptr(v))
                keep.append(v)
        for name in ("norm_attn", "norm_ffn"):
            if lw.get(name) is not None:
                setattr(arr[i], name, _ptr(lw[name]))
                keep.append(lw[name])
    return arr, keep


def head_weight_struct(head: Dict[str, object]):
    """{"norm": bf16 [H], "lm": Int4Matrix [vocab][H]} -> (ctypes struct, tensors kept alive)."""
    lm = head["lm"]
    if not hasattr(lm, "packed"):
        raise KvrError(-6, "the output head needs int4 weights")
    st = KvrHeadWeights(_ptr(head["norm"]), _ptr(lm.packed), _ptr(lm.scales), int(lm.packed.shape[0]))
    return st, [head["norm"], lm.packed, lm.scales]


def _i32(tokens) -> ctypes.Array:
    """Token ids as a C int32 array (at least one element) that shares memory
    with one contiguous copy: an int32 numpy array is passed as it is, a list
    goes through array('i') (a per-element ctypes constructor costs ~60 us for
    254 tokens, on the path between a match and the prefill it decides)."""
    if isinstance(tokens, np.ndarray):
        a = np.ascontiguousarray(tokens, dtype=np.int32)
        if a.size == 0:
            a = np.zeros(1, np.int32)
        elif not a.flags.writeable:   # from_buffer needs a writable buffer
            a = a.copy()
        return (ctypes.c_int32 * a.size).from_buffer(a)
    a = array.array("i", tokens)
    if not a:
        a.append(0)
    return (ctypes.c_int32 * len(a)).from_buffer(a)


assert array.array("i").itemsize == 4, "C int must be 32 bits"


class Kvr:
    """One libkvr context over a torch-allocated KV arena and scratch area."""

    def __init__(self, cfg: KvrConfig, device="cuda", arena_slots: Optional[int] = None):
        self.lib = load_library()
        self.cfg = cfg
        self.device = torch.device(device)
        n = arena_slots if arena_slots is not None else max(cfg.n_slots, 1)
        ab = self.lib.kvr_arena_bytes(ctypes.byref(cfg), n)
        sb = self.lib.kvr_scratch_bytes(ctypes.byref(cfg))
        if ab == 0 or sb == 0:
            raise KvrError(-1, "invalid configuration")
        self.arena = torch.empty(ab, dtype=torch.uint8, device=self.device)
        self.scratch = torch.empty(sb, dtype=torch.uint8, device=self.device)
        ctx = ctypes.c_void_p()
        rc = self.lib.kvr_ctx_create(ctypes.byref(cfg), self.arena.data_ptr(), ab,
                                     self.scratch.data_ptr(), sb, ctypes.byref(ctx))
        if rc != KVR_OK:
            raise KvrError(rc, "kvr_ctx_create failed")
        self.ctx = ctx
        self._weights_cache = None

    # -------------------------------------------------------------- helpers
    def close(self):
        if getattr(self, "ctx", None):
            self.lib.kvr_ctx_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc: int):
        if rc != KVR_OK:
            raise KvrError(rc, self.lib.kvr_last_error(self.ctx).decode())

    @staticmethod
    def _stream(stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        return ctypes.c_void_p(s.cuda_stream)

    def weights(self, layers):
        arr, keep = layer_weight_structs(layers)
        return arr, keep

    # -------------------------------------------------------------- C ABI
    def kvr_ctx_info(self) -> Tuple[int, int, int]:
        g, r, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        self._check(self.lib.kvr_ctx_info(self.ctx, ctypes.byref(g), ctypes.byref(r), ctypes.byref(c)))
        return g.value, r.value, c.value

    def kvr_slot_match(self, tokens, stream=None) -> Tuple[int, int]:
        s, r = ctypes.c_int(), ctypes.c_int()
        self._check(self.lib.kvr_slot_match(self.ctx, _i32(tokens), len(tokens), ctypes.byref(s),
                                            ctypes.byref(r), self._stream(stream)))
        return s.value, r.value

    def kvr_slot_match_static(self, tokens, stream=None) -> Tuple[int, int]:
        """kvr_slot_match staged in the library's fixed device array (no caller scratch)."""
        s, r = ctypes.c_int(), ctypes.c_int()
        self._check(self.lib.kvr_slot_match_static(self.ctx, _i32(tokens), len(tokens),
                                                   ctypes.byref(s), ctypes.byref(r),
                                                   self._stream(stream)))
        return s.value, r.value

    def kvr_slot_truncate(self, slot: int, new_len: int):
        self._check(self.lib.kvr_slot_truncate(self.ctx, slot, new_len))

    def kvr_slot_len(self, slot: int) -> int:
        n = ctypes.c_int()
        self._check(self.lib.kvr_slot_len(self.ctx, slot, ctypes.byref(n)))
        return n.value

    def kvr_slot_tokens(self, slot: int) -> List[int]:
        n = self.kvr_slot_len(slot)
        buf = (ctypes.c_int32 * max(n, 1))()
        self._check(self.lib.kvr_slot_tokens(self.ctx, slot, buf, n))
        return list(buf[:n])

    def kvr_slot_assign(self, slot: int, tokens, stream=None):
        self._check(self.lib.kvr_slot_assign(self.ctx, slot, _i32(tokens), len(tokens),
                                             self._stream(stream)))

    def kvr_slot_kv(self, slot: int, layer: int) -> Tuple[torch.Tensor, torch.Tensor]:
        """K view [Hkv][capacity][head_dim] and V view [Hkv][head_dim][capacity] (V is
        stored transposed) of one slot and layer, bf16."""
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        self._check(self.lib.kvr_slot_kv(self.ctx, slot, layer, ctypes.byref(k), ctypes.byref(v)))
        c = self.cfg
        n = c.n_kv_heads * c.capacity * c.head_dim
        flat = self.arena.view(torch.bfloat16)
        base = self.arena.data_ptr()
        ko, vo = (k.value - base) // 2, (v.value - base) // 2
        return (flat[ko:ko + n].view(c.n_kv_heads, c.capacity, c.head_dim),
                flat[vo:vo + n].view(c.n_kv_heads, c.head_dim, c.capacity))

    def _rows_call(self, fn, slot, tokens, hidden, weights, out, stream):
        arr = weights[0] if isinstance(weights, tuple) else weights
        m = len(tokens)
        assert hidden.dtype == torch.bfloat16 and hidden.is_cuda and hidden.is_contiguous()
        assert hidden.shape == (m, self.cfg.hidden)
        if out is None:
            out = torch.empty((m, self.cfg.hidden), dtype=torch.bfloat16, device=self.device)
        self._check(fn(self.ctx, slot, _i32(tokens), m, hidden.data_ptr(), arr, out.data_ptr(),
                       self._stream(stream)))
        return out

    def kvr_prefill_suffix(self, slot, tokens, hidden, weights, out=None, stream=None):
        return self._rows_call(self.lib.kvr_prefill_suffix, slot, tokens, hidden, weights, out, stream)

    def kvr_verify(self, slot, tokens, hidden, weights, out=None, stream=None):
        return self._rows_call(self.lib.kvr_verify, slot, tokens, hidden, weights, out, stream)

    def kvr_verify_accept(self, slot, tokens, hidden, weights, head, out=None, stream=None):
        """Verify [t0, d1 .. dk] and take the greedy decision.  Returns
        (next_tokens: the argmax of every row, accepted: the drafts kept)."""
        arr = weights[0] if isinstance(weights, tuple) else weights
        hs, _keep = head_weight_struct(head)
        m = len(tokens)
        assert hidden.dtype == torch.bfloat16 and hidden.is_cuda and hidden.is_contiguous()
        assert hidden.shape == (m, self.cfg.hidden)
        nxt = (ctypes.c_int32 * max(m, 1))()
        acc = ctypes.c_int()
        self._check(self.lib.kvr_verify_accept(self.ctx, slot, _i32(tokens), m, hidden.data_ptr(), arr,
                                               ctypes.byref(hs), _ptr(out), nxt, ctypes.byref(acc),
                                               self._stream(stream)))
        return list(nxt[:m]), acc.value

    def kvr_verify_accept_batch(self, slots, token_lists, hidden, weights, head, out=None, stream=None):
        """Greedy verification of conversation j's rows token_lists[j] on slot
        slots[j], all in one call.  Returns (per conversation: the argmax of
        each of its rows, the drafts kept)."""
        arr = weights[0] if isinstance(weights, tuple) else weights
        hs, _keep = head_weight_struct(head)
        lens = [len(t) for t in token_lists]
        m = sum(lens)
        assert hidden.dtype == torch.bfloat16 and hidden.is_cuda and hidden.is_contiguous()
        assert hidden.shape == (m, self.cfg.hidden)
        n = len(slots)
        slots_c = (ctypes.c_int * max(n, 1))(*[int(s) for s in slots])
        lens_c = (ctypes.c_int * max(n, 1))(*lens)
        nxt = (ctypes.c_int32 * max(m, 1))()
        acc = (ctypes.c_int * max(n, 1))()
        self._check(self.lib.kvr_verify_accept_batch(self.ctx, n, slots_c, lens_c, _i32(sum(token_lists, [])),
                                                     hidden.data_ptr(), arr, ctypes.byref(hs), _ptr(out),
                                                     nxt, acc, self._stream(stream)))
        out_next, at = [], 0
        for L in lens:
            out_next.append(list(nxt[at:at + L]))
            at += L
        return out_next, list(acc[:n])

    def kvr_prefill_batch(self, slots, token_lists, hidden, weights, out=None, stream=None):
        """Conversation j's rows token_lists[j] (hidden rows concatenated in the
        same order) appended to slot slots[j]; returns the rows' outputs."""
        arr = weights[0] if isinstance(weights, tuple) else weights
        lens = [len(t) for t in token_lists]
        m = sum(lens)
        assert hidden.dtype == torch.bfloat16 and hidden.is_cuda and hidden.is_contiguous()
        assert hidden.shape == (m, self.cfg.hidden)
        if out is None:
            out = torch.empty((m, self.cfg.hidden), dtype=torch.bfloat16, device=self.device)
        n = len(slots)
        slots_c = (ctypes.c_int * max(n, 1))(*[int(s) for s in slots])
        lens_c = (ctypes.c_int * max(n, 1))(*lens)
        self._check(self.lib.kvr_prefill_batch(self.ctx, n, slots_c, lens_c, _i32(sum(token_lists, [])),
                                               hidden.data_ptr(), arr, out.data_ptr(), self._stream(stream)))
        return out

    def kvr_selftest_wait(self, stream=None):
        self._check(self.lib.kvr_selftest_wait(self.ctx, self._stream(stream)))

    def kvr_slot_spill(self, slot: int, model_tag: int = 0, stream=None, sync: bool = True) -> torch.Tensor:
        """The slot's record in pinned host memory (uint8); complete once the
        stream has passed the copies (sync=True waits for it)."""
        n = self.lib.kvr_slot_spill_bytes(self.ctx, slot)
        if n == 0:
            raise KvrError(-1, f"bad slot {slot}")
        rec = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        st = self._stream(stream)
        self._check(self.lib.kvr_slot_spill(self.ctx, slot, model_tag, rec.data_ptr(), n, st))
        if sync:
            (stream if stream is not None else torch.cuda.current_stream()).synchronize()
        return rec

    def kvr_slot_restore(self, slot: int, record: torch.Tensor, model_tag: int = 0, stream=None,
                         sync: bool = True):
        assert record.dtype == torch.uint8 and record.device.type == "cpu" and record.is_contiguous()
        self._check(self.lib.kvr_slot_restore(self.ctx, slot, model_tag, record.data_ptr(), record.numel(),
                                              self._stream(stream)))
        if sync:
            (stream if stream is not None else torch.cuda.current_stream()).synchronize()

    def kvr_prefill_branches(self, slot, lens, tokens, hidden, weights, out=None, stream=None):
        arr = weights[0] if isinstance(weights, tuple) else weights
        m = hidden.shape[0]
        assert sum(lens) == m == len(tokens)
        if out is None:
            out = torch.empty((m, self.cfg.hidden), dtype=torch.bfloat16, device=self.device)
        lens_c = (ctypes.c_int * len(lens))(*[int(x) for x in lens])
        self._check(self.lib.kvr_prefill_branches(self.ctx, slot, len(lens), lens_c, _i32(tokens),
                                                  hidden.data_ptr(), arr, out.data_ptr(),
                                                  self._stream(stream)))
        return out

    def kvr_sync_status(self, stream=None):
        self._check(self.lib.kvr_sync_status(self.ctx, self._stream(stream)))

    def kvr_trace_set(self, buf: Optional[torch.Tensor]):
        """buf: float32 device tensor [n_layers + 1][max_rows][hidden], or None to clear."""
        if buf is None:
            self._check(self.lib.kvr_trace_set(self.ctx, None, 0))
        else:
            assert buf.dtype == torch.float32 and buf.is_cuda and buf.is_contiguous()
            self._check(self.lib.kvr_trace_set(self.ctx, buf.data_ptr(), buf.numel() * 4))
        self._trace = buf

    def kvr_profile_enable(self, on: bool):
        self._check(self.lib.kvr_profile_enable(self.ctx, 1 if on else 0))

    def kvr_profile_read(self):
        ms = (ctypes.c_float * 4)()
        n = (ctypes.c_int * 4)()
        self._check(self.lib.kvr_profile_read(self.ctx, ms, n))
        return list(ms), list(n)

    def kvr_profile_launches(self, max_n: int = 65536):
        """[(class, ms)] of the launches recorded since the last kvr_profile_read."""
        cls = (ctypes.c_int * max_n)()
        ms = (ctypes.c_float * max_n)()
        n = ctypes.c_int()
        self._check(self.lib.kvr_profile_launches(self.ctx, cls, ms, max_n, ctypes.byref(n)))
        return [(cls[i], ms[i]) for i in range(min(n.value, max_n))]
