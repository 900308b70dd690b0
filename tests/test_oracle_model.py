"""Pins of the oracle's decoder layer (no GPU): closed forms, invariants and
the split / branch equalities the pages fix."""
import numpy as np
import pytest

import workloads
from oracle import model
from oracle.model import Dims, SlotKV, attend, rmsnorm, rope, softmax
from oracle.numerics import round_bf16, silu
from conftest import oracle_dims, oracle_weights, read_fixture


# ---------------------------------------------------------------- attention

def test_constant_v_per_kv_head_gives_that_constant(rng):
    # Hq = 6, Hkv = 3: head h must read KV head h // 2
    K = rng.standard_normal((3, 20, 16))
    V = np.empty((3, 20, 16))
    consts = [1.5, -2.25, 4.0]
    for j, c in enumerate(consts):
        V[j] = c
    q = rng.standard_normal((6, 16)) * 3
    o = attend(q, K, V, np.arange(13), group=2)
    for h in range(6):
        np.testing.assert_allclose(o[h], consts[h // 2], rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_visible_values(rng):
    K = rng.standard_normal((1, 30, 8))
    V = rng.standard_normal((1, 30, 8))
    vis = np.arange(17)
    o = attend(np.zeros((2, 8)), K, V, vis, group=2)
    np.testing.assert_allclose(o[0], V[0, :17].mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[1], V[0, :17].mean(axis=0), rtol=0, atol=1e-14)


def test_single_row_at_position_zero_sees_only_itself(rng):
    K = rng.standard_normal((2, 5, 8))
    V = rng.standard_normal((2, 5, 8))
    o = attend(rng.standard_normal((4, 8)), K, V, np.arange(1), group=2)
    np.testing.assert_array_equal(o[0], V[0, 0])
    np.testing.assert_array_equal(o[3], V[1, 0])


def test_two_key_softmax_closed_form():
    # scores a/sqrt(d) and 0 -> weight of key 0 is the logistic of a/sqrt(d)
    d, a = 16, 3.0
    K = np.zeros((1, 2, d)); K[0, 0, 0] = 1.0
    V = np.zeros((1, 2, d)); V[0, 0, :] = 1.0
    q = np.zeros((1, d)); q[0, 0] = a
    o = attend(q, K, V, np.arange(2), group=1)
    p0 = 1.0 / (1.0 + np.exp(-a / np.sqrt(d)))
    np.testing.assert_allclose(o[0], p0, rtol=1e-14)


def test_softmax_rows_sum_to_one(rng):
    for n in (1, 2, 7, 1000):
        s = rng.standard_normal(n) * 20
        p = softmax(s)
        assert abs(p.sum() - 1.0) <= 1e-12
        assert np.all(p >= 0)


def test_keys_outside_the_visible_set_do_not_matter(rng):
    K = rng.standard_normal((1, 40, 8)); V = rng.standard_normal((1, 40, 8))
    q = rng.standard_normal((1, 8))
    o1 = attend(q, K, V, np.arange(25), 1)
    K[:, 25:] = 99.0; V[:, 25:] = -99.0
    np.testing.assert_array_equal(o1, attend(q, K, V, np.arange(25), 1))


# ---------------------------------------------------------------- RoPE

def test_rope_worked_example():
    fx = read_fixture("rope_fixture.txt")
    x = np.array([float(v) for v in fx["x"]])[None, :]
    got = rope(x, int(fx["pos"][0]), float(fx["theta"][0]))[0]
    np.testing.assert_allclose(got, [float(v) for v in fx["out"]], rtol=1e-14)


def test_rope_position_zero_is_identity_and_preserves_norm(rng):
    x = rng.standard_normal((4, 128))
    np.testing.assert_array_equal(rope(x, 0, 1e6), x)
    y = rope(x, 1234, 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_scores_depend_on_position_difference_only(rng):
    q = rng.standard_normal((1, 64)); k = rng.standard_normal((1, 64))
    base = (rope(q, 100, 1e4) * rope(k, 37, 1e4)).sum()
    for t in (1, 50, 900):
        np.testing.assert_allclose((rope(q, 100 + t, 1e4) * rope(k, 37 + t, 1e4)).sum(), base,
                                   rtol=1e-10)


# ---------------------------------------------------------------- RMSNorm / FFN

def test_rmsnorm_invariants(rng):
    h = rng.standard_normal((3, 256)) * 7
    g = np.ones(256)
    a = rmsnorm(h, g, 1e-12)
    np.testing.assert_allclose(np.mean(a * a, axis=1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(rmsnorm(h * 13.0, g, 1e-12), a, rtol=1e-12)
    c = np.full((1, 8), -0.5)
    np.testing.assert_allclose(rmsnorm(c, np.ones(8), 1e-6), -0.5 / np.sqrt(0.25 + 1e-6), rtol=1e-14)
    gains = np.arange(1, 9, dtype=float)
    np.testing.assert_allclose(rmsnorm(c, gains, 0.0)[0], -gains, rtol=1e-14)


def _identity_ffn_layer(H, gate_scale, up_scale):
    eye = np.eye(H)
    return {"wq": np.zeros((H, H)), "wk": np.zeros((H, H)), "wv": np.zeros((H, H)),
            "wo": np.zeros((H, H)), "wg": gate_scale * eye, "wu": up_scale * eye, "wd": eye,
            "norm_attn": np.ones(H), "norm_ffn": np.ones(H)}


def test_ffn_closed_form_distinguishes_gate_and_up():
    # Wo = 0, Wg = 2I, Wu = I, Wd = I, h = c*1: b = bf16(c/sqrt(c^2+eps)),
    # out = h + bf16(silu(2b) * b)
    H, c, eps = 8, 0.75, 1e-6
    dims = Dims(H, 1, 1, H, H, False, 1e6, eps)
    W = _identity_ffn_layer(H, 2.0, 1.0)
    kv = SlotKV(1, 1, 4, H)
    out = model.layer(dims, W, np.full((1, H), c), kv.K[0], kv.V[0], model.plain_rows(0, 1))
    b = round_bf16(c / np.sqrt(c * c + eps))
    np.testing.assert_allclose(out, c + round_bf16(silu(2 * b) * b), rtol=1e-15)
    W2 = _identity_ffn_layer(H, 1.0, 2.0)
    out2 = model.layer(dims, W2, np.full((1, H), c), kv.K[0], kv.V[0], model.plain_rows(0, 1))
    np.testing.assert_allclose(out2, c + round_bf16(silu(b) * 2 * b), rtol=1e-15)
    assert abs(out2 - out).max() > 0.1


def test_zero_output_projections_make_the_layer_the_identity(rng):
    shape = workloads.SHAPES["small"]
    W = oracle_weights(shape, workloads.layer_weights(shape, 7, 0))
    W["wo"] = np.zeros_like(W["wo"]); W["wd"] = np.zeros_like(W["wd"])
    kv = SlotKV(1, shape.n_kv_heads, 64, shape.head_dim)
    h = rng.standard_normal((5, shape.hidden))
    out = model.layer(oracle_dims(shape), W, h, kv.K[0], kv.V[0], model.plain_rows(3, 5))
    np.testing.assert_array_equal(out, h)


# ---------------------------------------------------------------- split / branches

def _small_stack(name="small", seed=11):
    shape = workloads.SHAPES[name]
    lws = workloads.stack_weights(shape, seed)
    return shape, oracle_dims(shape), [oracle_weights(shape, lw) for lw in lws]


def test_whole_prompt_equals_prefix_then_suffix():
    shape, dims, W = _small_stack()
    toks = list(range(100, 160))
    x = workloads.bf16_to_f64(workloads.hidden_for_tokens(toks, shape.hidden, 5))
    kv_whole = SlotKV(shape.n_layers, shape.n_kv_heads, 64, shape.head_dim)
    whole = model.prefill(dims, W, kv_whole, x, 0)
    kv_split = SlotKV(shape.n_layers, shape.n_kv_heads, 64, shape.head_dim)
    model.prefill(dims, W, kv_split, x[:41], 0)
    suffix = model.prefill(dims, W, kv_split, x[41:], 41)
    np.testing.assert_array_equal(suffix, whole[41:])
    np.testing.assert_array_equal(kv_split.K[:, :, :60], kv_whole.K[:, :, :60])
    np.testing.assert_array_equal(kv_split.V[:, :, :60], kv_whole.V[:, :, :60])


def test_verify_rows_equal_one_row_steps():
    # m = k+1 rows at once == k+1 single-row steps (the one-token-short fix)
    shape, dims, W = _small_stack("small_d128", 3)
    toks = list(range(7, 27))
    x = workloads.bf16_to_f64(workloads.hidden_for_tokens(toks, shape.hidden, 2))
    kv_a = SlotKV(shape.n_layers, shape.n_kv_heads, 32, shape.head_dim)
    model.prefill(dims, W, kv_a, x[:16], 0)
    kv_b = SlotKV(shape.n_layers, shape.n_kv_heads, 32, shape.head_dim)
    kv_b.K[:] = kv_a.K; kv_b.V[:] = kv_a.V
    batch = model.prefill(dims, W, kv_a, x[16:], 16)
    steps = np.concatenate([model.prefill(dims, W, kv_b, x[16 + i:17 + i], 16 + i) for i in range(4)])
    np.testing.assert_array_equal(batch, steps)


def test_branches_equal_separate_runs():
    shape, dims, W = _small_stack()
    P, lens = 23, [5, 9, 1, 7]
    state = workloads.bf16_to_f64(workloads.hidden_for_tokens(list(range(P)), shape.hidden, 9))
    qs = [workloads.bf16_to_f64(workloads.hidden_for_tokens(list(range(500 + 10 * b, 500 + 10 * b + n)),
                                                            shape.hidden, 9)) for b, n in enumerate(lens)]
    kv = SlotKV(shape.n_layers, shape.n_kv_heads, 64, shape.head_dim)
    model.prefill(dims, W, kv, state, 0)
    base_K, base_V = kv.K.copy(), kv.V.copy()
    batched = model.prefill_branches(dims, W, kv, np.concatenate(qs), P, lens)
    off = 0
    for b, n in enumerate(lens):
        kv_b = SlotKV(shape.n_layers, shape.n_kv_heads, 64, shape.head_dim)
        kv_b.K[:] = base_K; kv_b.V[:] = base_V
        alone = model.prefill(dims, W, kv_b, qs[b], P)
        np.testing.assert_array_equal(batched[off:off + n], alone)
        off += n


def test_attn_only_layer_structure(rng):
    # attention-only layer (the tiny config): out = bf16(bf16(attn) Wo^T); with
    # constant V per head the attention output is that constant exactly
    shape = workloads.SHAPES["tiny"]
    dims = oracle_dims(shape)
    H, d = shape.hidden, shape.head_dim
    W = {"wq": rng.standard_normal((shape.q_dim, H)) * 0.02, "wk": rng.standard_normal((d, H)) * 0.02,
         "wv": np.zeros((d, H)), "wo": rng.standard_normal((H, shape.q_dim)) * 0.02}
    kv = SlotKV(1, 1, 16, d)
    kv.V[0, 0, :10] = 0.5
    x = rng.standard_normal((3, H))
    out = model.layer(dims, W, x, kv.K[0], kv.V[0], model.plain_rows(10, 3))
    # new rows' V = x Wv^T = 0, so output rows mix 0.5 and 0 with softmax weights
    # and the output is Wo applied to a per-head scalar times ones
    assert out.shape == (3, H)
    W["wv"] = np.zeros((d, H)); kv.V[0, 0, :10] = 0.0
    out0 = model.layer(dims, W, x, kv.K[0], kv.V[0], model.plain_rows(10, 3))
    np.testing.assert_array_equal(out0, 0.0)


@pytest.mark.parametrize("name", ["small", "small_attn"])
def test_layer_rows_equals_layer_on_selected_rows(name, rng):
    shape = workloads.SHAPES[name]
    dims = oracle_dims(shape)
    W = oracle_weights(shape, workloads.layer_weights(shape, 4, 0))
    m, P = 11, 9
    h = rng.standard_normal((m, shape.hidden))
    kv1 = SlotKV(1, shape.n_kv_heads, 32, shape.head_dim)
    kv1.K[0][:, :P] = round_bf16(rng.standard_normal((shape.n_kv_heads, P, shape.head_dim)))
    kv1.V[0][:, :P] = round_bf16(rng.standard_normal((shape.n_kv_heads, P, shape.head_dim)))
    kv2 = SlotKV(1, shape.n_kv_heads, 32, shape.head_dim)
    kv2.K[:] = kv1.K; kv2.V[:] = kv1.V
    full = model.layer(dims, W, h, kv1.K[0], kv1.V[0], model.plain_rows(P, m))
    sel = [0, 4, 10]
    part = model.layer_rows(dims, W, h, kv2.K[0], kv2.V[0], model.plain_rows(P, m), sel)
    np.testing.assert_array_equal(part, full[sel])
    np.testing.assert_array_equal(kv2.K, kv1.K)
    np.testing.assert_array_equal(kv2.V, kv1.V)


# ---------------------------------------------------------------- head and greedy acceptance

def test_greedy_accept_hand_worked():
    acc = model.greedy_accept
    # rows [t0, d1, d2, d3]; argmax[j] is the model's next token after row j
    assert acc([5, 7, 9, 11], [7, 9, 11, 3]) == 3          # every draft agrees
    assert acc([5, 7, 9, 11], [8, 9, 11, 3]) == 0          # the first draft is rejected
    assert acc([5, 7, 9, 11], [7, 9, 2, 3]) == 2           # d3 differs from argmax of row 2
    assert acc([5, 7, 9, 11], [7, 1, 11, 3]) == 1          # later agreement does not count
    assert acc([5], [4]) == 0                              # m = 1: nothing to accept


def test_greedy_argmax_takes_lowest_index_on_ties():
    logits = np.array([[1.0, 3.0, 3.0, -1.0], [0.0, 0.0, 0.0, 0.0]])
    assert model.greedy_argmax(logits).tolist() == [1, 0]


def test_head_with_identity_lm_ranks_the_normed_stream(rng):
    dims = Dims(64, 4, 2, 16, 128, False)
    h = rng.standard_normal((3, 64)) * 7.0
    gain = np.ones(64)
    logits = model.head_logits(dims, h, gain, np.eye(64))
    normed = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + dims.rms_eps)
    np.testing.assert_array_equal(logits, round_bf16(normed))
    assert (model.greedy_argmax(logits) == np.argmax(h, axis=-1)).all()


def test_head_single_row_is_its_dot_product(rng):
    dims = Dims(32, 4, 2, 8, 64, False)
    h = rng.standard_normal((2, 32))
    gain = rng.uniform(0.5, 1.5, 32)
    w = np.zeros((10, 32))
    w[6] = rng.standard_normal(32)
    logits = model.head_logits(dims, h, gain, w)
    b = round_bf16(rmsnorm(h, gain, dims.rms_eps))
    assert np.count_nonzero(logits[:, [0, 1, 2, 3, 4, 5, 7, 8, 9]]) == 0
    np.testing.assert_allclose(logits[:, 6], b @ w[6], rtol=0, atol=1e-12)
