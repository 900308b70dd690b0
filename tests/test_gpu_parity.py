"""CUDA path vs the oracle, through the C ABI (needs a GB300).

Tolerance (the stated bf16 bar): |gpu - oracle| <= 1e-2 + 2e-2*|oracle| for
every element of every compared output and of the K/V written to the slot;
slot choice, reused counts and lengths are exact.
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import oracle_dims, oracle_weights
from oracle import model as om
from oracle.slots import SlotTable

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))   # NaN fails
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} out of tolerance, max err "
                           f"{err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def make(shape_name, n_slots, cap, max_rows, seed=21, threshold=True, scales="fp16"):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES[shape_name]
    lws = workloads.stack_weights(shape, seed, scales=scales)
    kv = Kvr(config_for_shape(shape, n_slots, cap, max_rows, threshold), device="cuda")
    gw = workloads.weights_to(lws, "cuda")
    w = kv.weights(gw)
    W = [oracle_weights(shape, lw) for lw in lws]
    return shape, kv, w, W, gw


def hidden(tokens, shape, seed=5):
    return workloads.hidden_for_tokens(tokens, shape.hidden, seed)


def slot_kv_f64(kv, slot, layer, n):
    """K, V of a slot as [Hkv][n][d] (V is stored transposed in the arena)."""
    k, v = kv.kvr_slot_kv(slot, layer)
    return workloads.bf16_to_f64(k[:, :n]), workloads.bf16_to_f64(v[:, :, :n].transpose(1, 2))


# --------------------------------------------------------------------------- config 1

def test_tiny_config_exact():
    """Config 1: 2 slots of 256, slot0 96 tokens, slot1 64, prompt shares 90 with slot0."""
    shape = workloads.SHAPES["tiny"]
    seed = workloads.config_seed(1)
    tk = workloads.tiny_tokens(seed)
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    lw = workloads.layer_weights(shape, seed, 0)
    kv = Kvr(config_for_shape(shape, 2, 256, 128), device="cuda")
    w = kv.weights(workloads.weights_to([lw], "cuda"))
    for s, name in ((0, "slot0"), (1, "slot1")):
        assert kv.kvr_slot_match(tk[name]) == (s, 0)
        kv.kvr_prefill_suffix(s, tk[name], hidden(tk[name], shape, seed).cuda(), w)
    assert kv.kvr_slot_match(tk["prompt"]) == (0, 90)
    assert kv.kvr_slot_len(0) == 90
    suffix = tk["prompt"][90:]
    out = kv.kvr_prefill_suffix(0, suffix, hidden(suffix, shape, seed).cuda(), w)
    kv.kvr_sync_status()
    assert kv.kvr_slot_len(0) == 120 and kv.kvr_slot_tokens(0) == tk["prompt"]

    dims = oracle_dims(shape)
    W = [oracle_weights(shape, lw)]
    cache = om.SlotKV(1, 1, 256, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(hidden(tk["prompt"], shape, seed)), 0)
    close(workloads.bf16_to_f64(out), whole[90:], "tiny suffix output")
    k, v = slot_kv_f64(kv, 0, 0, 120)
    close(k, cache.K[0][:, :120], "tiny K")
    close(v, cache.V[0][:, :120], "tiny V")


# --------------------------------------------------------------------------- stacks

@pytest.mark.parametrize("shape_name,P,ms,cap", [
    ("small", 70, [1, 3, 8, 9, 17, 40, 130], 256),
    ("small_d128", 45, [1, 5, 16, 33, 100], 256),
    ("small_bf16", 33, [2, 11, 35], 256),
    ("small", 150, [300], 512),
    ("small_q4k", 70, [1, 3, 9, 17, 40, 130], 256),   # K-quant: GEMV at 8/16/32 tokens, tcgen05 GEMM
    ("wide", 40, [1, 9, 40], 256),                     # hidden 4352: row kernels past 4096 elements
])
def test_suffix_prefill_matches_oracle(shape_name, P, ms, cap):
    shape, kv, w, W, _ = make(shape_name, 2, cap, min(cap, 320))
    dims = oracle_dims(shape)
    toks = list(range(1000, 1000 + P + max(ms)))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, cap, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)

    assert kv.kvr_slot_match(toks[:P]) == (0, 0)
    pre = kv.kvr_prefill_suffix(0, toks[:P], x[:P].cuda(), w)
    close(workloads.bf16_to_f64(pre), whole[:P], f"{shape_name} prefix rows")
    for m in ms:
        kv.kvr_slot_truncate(0, P)
        out = kv.kvr_prefill_suffix(0, toks[P:P + m], x[P:P + m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[P:P + m], f"{shape_name} m={m}")
        for l in range(shape.n_layers):
            k, v = slot_kv_f64(kv, 0, l, P + m)
            close(k, cache.K[l][:, :P + m], f"{shape_name} m={m} K layer {l}")
            close(v, cache.V[l][:, :P + m], f"{shape_name} m={m} V layer {l}")
    assert kv.kvr_slot_len(0) == P + ms[-1]


@pytest.mark.parametrize("shape_name", ["small", "small_q4k"])
def test_many_rows_on_the_gemv_match_oracle(monkeypatch, shape_name):
    """KVR_FORCE_GEMV=1 keeps every m on the GEMV (32-row passes) and the split-KV
    attention: the residual epilogue and the RMSNorm launch then span passes."""
    monkeypatch.setenv("KVR_FORCE_GEMV", "1")
    shape, kv, w, W, _ = make(shape_name, 1, 256, 128)
    monkeypatch.delenv("KVR_FORCE_GEMV")
    dims = oracle_dims(shape)
    P = 50
    toks = list(range(3000, 3000 + P + 70))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    kv.kvr_slot_match(toks[:1])
    pre = kv.kvr_prefill_suffix(0, toks[:P], x[:P].cuda(), w)
    close(workloads.bf16_to_f64(pre), whole[:P], f"{shape_name} GEMV prefix rows")
    for m in (1, 40, 70):
        kv.kvr_slot_truncate(0, P)
        out = kv.kvr_prefill_suffix(0, toks[P:P + m], x[P:P + m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[P:P + m], f"{shape_name} GEMV m={m}")
        for l in range(shape.n_layers):
            k, v = slot_kv_f64(kv, 0, l, P + m)
            close(k, cache.K[l][:, :P + m], f"{shape_name} GEMV m={m} K layer {l}")
            close(v, cache.V[l][:, :P + m], f"{shape_name} GEMV m={m} V layer {l}")


@pytest.mark.parametrize("combine", ["0", "1"])
@pytest.mark.parametrize("shape_name", ["small", "small_d128"])
def test_split_kv_merge_matches_oracle(monkeypatch, shape_name, combine):
    """A 700-token prefix gives the small-m split-KV kernel several key splits per
    KV head.  With at most four rows per KV head (m = 1 here: G = 4 and 3) the
    last split of each (row tile, KV head) merges them; more rows, or
    KVR_ATTN_COMBINE=1, leave the merge to the combine launch.  Both against
    the oracle, with the new rows' K/V."""
    monkeypatch.setenv("KVR_ATTN_COMBINE", combine)
    shape, kv, w, W, _ = make(shape_name, 1, 1024, 256)
    monkeypatch.delenv("KVR_ATTN_COMBINE")
    dims = oracle_dims(shape)
    P = 700
    toks = list(range(2000, 2000 + P + 8))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 1024, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    kv.kvr_slot_match(toks[:1])
    for a in range(0, P, 256):
        b = min(P, a + 256)
        kv.kvr_prefill_suffix(0, toks[a:b], x[a:b].cuda(), w)
    for m in (1, 3, 8):
        kv.kvr_slot_truncate(0, P)
        out = kv.kvr_prefill_suffix(0, toks[P:P + m], x[P:P + m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[P:P + m], f"{shape_name} merge {combine} m={m}")
        for l in range(shape.n_layers):
            k, v = slot_kv_f64(kv, 0, l, P + m)
            close(k[:, P:], cache.K[l][:, P:P + m], f"{shape_name} m={m} new K layer {l}")
            close(v[:, P:], cache.V[l][:, P:P + m], f"{shape_name} m={m} new V layer {l}")


@pytest.mark.parametrize("shape_name", ["small", "small_q4k"])
def test_small_m_on_the_tensor_core_gemm_matches_oracle(monkeypatch, shape_name):
    """KVR_FORCE_GEMM=1 sends every m to the tcgen05 GEMM (N = 16 for up to 16 rows)."""
    monkeypatch.setenv("KVR_FORCE_GEMM", "1")
    shape, kv, w, W, _ = make(shape_name, 2, 256, 64)
    monkeypatch.delenv("KVR_FORCE_GEMM")
    dims = oracle_dims(shape)
    toks = list(range(900, 900 + 60))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    kv.kvr_slot_match(toks[:40])
    kv.kvr_prefill_suffix(0, toks[:40], x[:40].cuda(), w)
    for m in (1, 5, 17):
        kv.kvr_slot_truncate(0, 40)
        out = kv.kvr_prefill_suffix(0, toks[40:40 + m], x[40:40 + m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[40:40 + m], f"{shape_name} m={m} on the GEMM")


def test_five_bit_scales_named_case():
    """The named extra input case: scales with at most 5 significant bits, where
    every code*scale is exactly a bf16 (and fp16) number, through the GEMV
    (m = 3) and the tcgen05 GEMM (m = 40)."""
    shape, kv, w, W, _ = make("small", 1, 256, 128, scales="5bit")
    dims = oracle_dims(shape)
    toks = list(range(4000, 4000 + 120))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    kv.kvr_slot_match(toks[:1])
    pre = kv.kvr_prefill_suffix(0, toks[:70], x[:70].cuda(), w)
    close(workloads.bf16_to_f64(pre), whole[:70], "5-bit scales, 70 rows")
    for m in (3, 40):
        kv.kvr_slot_truncate(0, 70)
        out = kv.kvr_prefill_suffix(0, toks[70:70 + m], x[70:70 + m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[70:70 + m], f"5-bit scales m={m}")


@pytest.mark.parametrize("m", [3, 40])
def test_swapped_norm_gains_are_caught(m):
    """The two RMSNorm gains of a layer are distinct bf16 draws in [0.5, 1.5):
    the GPU output matches the oracle with the gains in place and fails the
    same bound against an oracle whose first layer has them swapped (the
    mistake is planted in the oracle's weights, on the CPU).  m = 3 takes the
    GEMV path, m = 40 the tcgen05 GEMM and its row-wise norms."""
    shape, kv, w, W, _ = make("small", 1, 256, 64)
    dims = oracle_dims(shape)
    toks = list(range(6000, 6000 + 50 + m))
    x = hidden(toks, shape)
    kv.kvr_slot_match(toks[:1])
    kv.kvr_prefill_suffix(0, toks[:50], x[:50].cuda(), w)
    out = workloads.bf16_to_f64(kv.kvr_prefill_suffix(0, toks[50:], x[50:].cuda(), w))
    kv.kvr_sync_status()
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    ref = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)[50:]
    close(out, ref, f"gains in place m={m}")
    Ws = [dict(lw) for lw in W]
    Ws[0]["norm_attn"], Ws[0]["norm_ffn"] = W[0]["norm_ffn"], W[0]["norm_attn"]
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    swapped = om.prefill(dims, Ws, cache, workloads.bf16_to_f64(x), 0)[50:]
    with pytest.raises(AssertionError):
        close(out, swapped, f"gains swapped m={m}")


def peaked_kv(n_kv_heads, P, d, alpha_max, seed):
    """Cached K/V for a sharply peaked, steadily sharpening softmax: key j is
    alpha_j * z_j with z_j ~ N(0, I) and alpha_j rising linearly from
    0.05*alpha_max to alpha_max over the prefix, so a row's scores spread
    wider block after block and its running maximum keeps growing; V ~ N(0, 1).
    Both rounded to bf16, [Hkv][P][d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.standard_normal((n_kv_heads, P, d), dtype=np.float32)
    alpha = (alpha_max * (0.05 + 0.95 * np.arange(P) / max(P - 1, 1))).astype(np.float32)
    v = rng.standard_normal((n_kv_heads, P, d), dtype=np.float32)
    return workloads.to_bf16(z * alpha[None, :, None]), workloads.to_bf16(v)


@pytest.mark.parametrize("splits", ["0", "2"])
@pytest.mark.parametrize("combine", ["0", "1"])
@pytest.mark.parametrize("shape_name,P,alpha,ms", [
    ("small_attn", 1000, 40.0, [1, 3, 8, 40]),     # split-KV up to 24 rows, tcgen05 from 25
    ("qwen7b_attn", 2000, 16.0, [1, 4, 16, 64]),   # split-KV up to 13 rows, tcgen05 from 14
])
def test_peaked_attention_matches_oracle(monkeypatch, shape_name, P, alpha, ms, combine, splits):
    """Scores with std >= 10 whose row maximum grows across the prefix: the
    tcgen05 kernel must move its lazy reference maximum (and rescale O) many
    times, and the split-KV kernel must merge splits whose maxima differ by
    many units, by the last split (one row per warp) or by the combine launch
    (KVR_ATTN_COMBINE=1).  KVR_ATTN_SPLITS=2 runs the tcgen05 kernel with the
    two key splits of the turn-9 shape instead of its default four here.
    Cached K/V given through kvr_slot_kv."""
    monkeypatch.setenv("KVR_ATTN_COMBINE", combine)
    monkeypatch.setenv("KVR_ATTN_SPLITS", splits)
    shape, kv, w, W, _ = make(shape_name, 2, 2176, 64, seed=workloads.config_seed(5))
    monkeypatch.delenv("KVR_ATTN_COMBINE")
    monkeypatch.delenv("KVR_ATTN_SPLITS")
    dims = oracle_dims(shape)
    kk, vv = peaked_kv(shape.n_kv_heads, P, shape.head_dim, alpha, 91)
    k, v = kv.kvr_slot_kv(1, 0)
    k[:, :P] = kk.cuda()
    v[:, :, :P] = vv.transpose(1, 2).cuda()
    kv.kvr_slot_assign(1, list(range(P)))
    cache = om.SlotKV(1, shape.n_kv_heads, 2176, shape.head_dim)
    cache.K[0][:, :P] = workloads.bf16_to_f64(kk)
    cache.V[0][:, :P] = workloads.bf16_to_f64(vv)
    new = list(range(9000, 9000 + max(ms)))
    x = hidden(new, shape)
    ref = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), P)
    # the inputs really are peaked: the last rows' score spread over the prefix
    q = workloads.bf16_to_f64(x[-1:]) @ W[0]["wq"].T
    s = (q.reshape(shape.n_q_heads, shape.head_dim)[0] @ cache.K[0][0, :P].T) / np.sqrt(shape.head_dim)
    assert s[-256:].std() >= 10.0 and s[-256:].max() > s[:256].max() + 20.0
    for m in ms:
        kv.kvr_slot_truncate(1, P)
        out = kv.kvr_prefill_suffix(1, new[:m], x[:m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), ref[:m], f"{shape_name} peaked m={m} combine={combine}")


def test_verify_then_truncate_equals_single_steps():
    shape, kv, w, W, _ = make("small", 2, 256, 64)
    dims = oracle_dims(shape)
    toks = list(range(50, 50 + 60))
    x = hidden(toks, shape)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    P = 52
    kv.kvr_slot_match(toks[:P])
    kv.kvr_prefill_suffix(0, toks[:P], x[:P].cuda(), w)
    # verify m = k+1 = 8 rows, accept 5 drafts -> keep P + 1 + 5
    out = kv.kvr_verify(0, toks[P:P + 8], x[P:P + 8].cuda(), w)
    close(workloads.bf16_to_f64(out), whole[P:P + 8], "verify rows")
    kv.kvr_slot_truncate(0, P + 1 + 5)
    assert kv.kvr_slot_len(0) == P + 6
    # the next step continues from the committed prefix exactly like one-row steps
    step = kv.kvr_prefill_suffix(0, toks[P + 6:P + 7], x[P + 6:P + 7].cuda(), w)
    close(workloads.bf16_to_f64(step), whole[P + 6:P + 7], "row after verify")
    for l in range(shape.n_layers):
        k, v = slot_kv_f64(kv, 0, l, P + 7)
        close(k, cache.K[l][:, :P + 7], "K after verify")
        close(v, cache.V[l][:, :P + 7], "V after verify")
    from prefix_reused_prefill_gb300 import KvrError
    with pytest.raises(KvrError):
        kv.kvr_verify(0, list(range(65)), torch.zeros(65, shape.hidden, dtype=torch.bfloat16).cuda(), w)


@pytest.mark.parametrize("P,lens", [(40, [5, 9, 1, 7]), (70, [30, 50, 1, 40])])
def test_branches_match_oracle_and_leave_checkpoint(P, lens):
    shape, kv, w, W, gw = make("small", 2, 256, 128)
    dims = oracle_dims(shape)
    state = list(range(7, 7 + P))
    qs = [list(range(2000 + 100 * b, 2000 + 100 * b + n)) for b, n in enumerate(lens)]
    xs = hidden(state, shape)
    xq = hidden(sum(qs, []), shape)
    kv.kvr_slot_match(state)
    kv.kvr_prefill_suffix(0, state, xs.cuda(), w)
    out = kv.kvr_prefill_branches(0, lens, sum(qs, []), xq.cuda(), w)
    kv.kvr_sync_status()
    assert kv.kvr_slot_len(0) == P and kv.kvr_slot_tokens(0) == state

    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    om.prefill(dims, W, cache, workloads.bf16_to_f64(xs), 0)
    ref = om.prefill_branches(dims, W, cache, workloads.bf16_to_f64(xq), P, lens)
    close(workloads.bf16_to_f64(out), ref, "branches")
    # each branch alone (truncate to the checkpoint, prefill) agrees too
    off = 0
    for b, n in enumerate(lens):
        alone = kv.kvr_prefill_suffix(0, qs[b], xq[off:off + n].cuda(), w)
        close(workloads.bf16_to_f64(alone), ref[off:off + n], f"branch {b} alone")
        kv.kvr_slot_truncate(0, P)
        off += n


def test_attention_only_7b_layer_with_given_kv():
    """Config-5 shape (one 7B attention + QKV/O layer), cached K/V given directly."""
    shape, kv, w, W, _ = make("qwen7b_attn", 4, 1024, 64, seed=workloads.config_seed(5))
    dims = oracle_dims(shape)
    P = 300
    kk, vv = workloads.random_kv(shape.n_kv_heads, P, shape.head_dim, 77)
    k, v = kv.kvr_slot_kv(2, 0)
    k[:, :P] = kk.cuda()
    v[:, :, :P] = vv.transpose(1, 2).cuda()
    state = list(range(P))
    kv.kvr_slot_assign(2, state)
    cache = om.SlotKV(1, shape.n_kv_heads, 1024, shape.head_dim)
    cache.K[0][:, :P] = workloads.bf16_to_f64(kk)
    cache.V[0][:, :P] = workloads.bf16_to_f64(vv)
    new = list(range(5000, 5064))
    x = hidden(new, shape)
    ref = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), P)
    for m in (1, 4, 16, 64):
        kv.kvr_slot_truncate(2, P)
        out = kv.kvr_prefill_suffix(2, new[:m], x[:m].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), ref[:m], f"7b attention layer m={m}")


# --------------------------------------------------------------------------- slot table

def test_match_kernel_and_policy_against_oracle():
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES["tiny"]
    rng = np.random.Generator(np.random.PCG64(99))
    for threshold in (True, False):
        for S in (1, 2, 3, 4):
            kv = Kvr(config_for_shape(shape, S, 64, 16, threshold), device="cuda")
            ref = SlotTable(S, 64, threshold)
            for trial in range(60):
                vocab = int(rng.integers(2, 4))
                for s in range(S):
                    if rng.random() < 0.85:
                        toks = rng.integers(0, vocab, size=int(rng.integers(0, 64))).tolist()
                        ref.assign(s, toks)
                        kv.kvr_slot_assign(s, toks)
                    elif ref.tokens[s] is not None:
                        # make the library forget the slot the same way: not possible
                        # directly, so give both the same (empty) content
                        ref.assign(s, [])
                        kv.kvr_slot_assign(s, [])
                prompt = rng.integers(0, vocab, size=int(rng.integers(1, 64))).tolist()
                want = ref.match(prompt)
                got = kv.kvr_slot_match(prompt)
                assert got == want, (threshold, S, trial)
                assert kv.kvr_slot_len(got[0]) == ref.length(want[0])
            kv.close()


def test_turn9_match_on_device():
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    tk = workloads.turn9_tokens()
    kv = Kvr(config_for_shape(workloads.SHAPES["tiny"], 4, 16384, 16), device="cuda")
    for s in range(4):
        kv.kvr_slot_assign(s, tk[f"slot{s}"])
    assert kv.kvr_slot_match(tk["prompt"]) == (0, 1668)
    assert kv.kvr_slot_len(0) == 1668


def test_reuse_off_and_granted_slots():
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES["tiny"]
    kv = Kvr(config_for_shape(shape, 0, 64, 16), device="cuda")
    kv.kvr_slot_assign(0, [1, 2, 3])
    assert kv.kvr_slot_match([1, 2, 3, 4]) == (0, 0)
    assert kv.kvr_ctx_info() == (1, 0, 64)
    # an arena with room for 2 of 4 requested slots grants 2
    kv2 = Kvr(config_for_shape(shape, 4, 64, 16), device="cuda", arena_slots=2)
    assert kv2.kvr_ctx_info() == (2, 4, 64)


def test_errors_leave_slots_unchanged():
    from prefix_reused_prefill_gb300 import KvrError
    shape, kv, w, W, _ = make("small", 2, 128, 64)
    toks = list(range(100))
    x = hidden(toks, shape).cuda()
    kv.kvr_slot_match(toks[:64])
    kv.kvr_prefill_suffix(0, toks[:64], x[:64].contiguous(), w)
    with pytest.raises(KvrError) as e:
        kv.kvr_prefill_suffix(0, toks[:64] + toks[:1], torch.zeros(65, shape.hidden, dtype=torch.bfloat16).cuda(), w)
    assert e.value.code == -2
    assert kv.kvr_slot_len(0) == 64
    with pytest.raises(KvrError) as e:
        kv.kvr_prefill_suffix(5, toks[:2], x[:2].contiguous(), w)
    assert e.value.code == -1
    with pytest.raises(KvrError) as e:
        kv.kvr_slot_truncate(0, 65)
    assert e.value.code == -1
    assert kv.kvr_slot_len(0) == 64
