"""Pins of the model-iteration oracle against library routines, closed forms and
the selective-batching invariants the pages state."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import model, padded, unbatched
from oracle.model import BatchItem, KVStore
from iteration_level_scheduling_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.TINY


def tiny_weights(seed=0, affine=True):
    return synth.make_weights(TINY, seed, random_affine=affine, std=0.05)


# --------------------------------------------------------------------------- #
# building blocks against torch CPU / closed forms
# --------------------------------------------------------------------------- #
def test_layer_norm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 33)) * 3 + 1
    g, b = rng.standard_normal(33), rng.standard_normal(33)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5)
    np.testing.assert_allclose(model.layer_norm(x, g, b), ref.numpy(), rtol=1e-12, atol=1e-12)
    # closed form: zero mean, unit (biased) variance before the affine map
    y = model.layer_norm(x, np.ones(33), np.zeros(33), eps=0.0)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(-1), 1, atol=1e-12)


def test_gelu_matches_torch_and_phi():
    x = np.linspace(-6, 6, 1001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="none").numpy()
    np.testing.assert_allclose(model.gelu(x), ref, rtol=1e-12, atol=1e-14)
    # GeLU(1) = Phi(1), the standard normal CDF at 1
    assert abs(model.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert model.gelu(np.array([0.0]))[0] == 0.0


def test_argmax_lowest_index_on_ties():
    v = np.array([0.0, 3.0, -1.0, 3.0, 3.0])
    assert model.argmax_lowest(v) == 1


def test_attention_matches_sdpa_prefill_and_cached():
    rng = np.random.default_rng(1)
    H, nh = 32, 4
    d = H // nh
    for ctx, n in [(0, 9), (5, 1), (6, 4)]:
        T = ctx + n
        q = rng.standard_normal((n, H))
        k = rng.standard_normal((T, H))
        v = rng.standard_normal((T, H))
        pos = ctx + np.arange(n)
        out = model.attention_one(q, k, v, pos, nh)
        qt = torch.from_numpy(q).view(n, nh, d).transpose(0, 1)
        kt = torch.from_numpy(k).view(T, nh, d).transpose(0, 1)
        vt = torch.from_numpy(v).view(T, nh, d).transpose(0, 1)
        mask = torch.from_numpy(np.arange(T)[None, :] <= pos[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
        np.testing.assert_allclose(out, ref.transpose(0, 1).reshape(n, H).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_closed_forms():
    H, nh = 16, 2
    rng = np.random.default_rng(2)
    v = rng.standard_normal((6, H))
    # identical keys: uniform weights over the visible prefix -> prefix mean of V
    k = np.tile(rng.standard_normal((1, H)), (6, 1))
    q = rng.standard_normal((3, H))
    pos = np.array([0, 2, 5])
    out = model.attention_one(q, k, v, pos, nh)
    for i, p in enumerate(pos):
        np.testing.assert_allclose(out[i], v[:p + 1].mean(0), rtol=1e-12, atol=1e-12)
    # one dominant key: output is that key's value row
    k2 = np.zeros((6, H))
    k2[3] = 1e3
    out = model.attention_one(np.ones((1, H)), k2, v, np.array([5]), nh)
    np.testing.assert_allclose(out[0], v[3], rtol=1e-9, atol=1e-9)


# --------------------------------------------------------------------------- #
# the whole block against torch's own pre-LN transformer layer
# --------------------------------------------------------------------------- #
def torch_reference_prefill(w, nh, tokens):
    H = w["tok_emb"].shape[1]
    F = w["layers"][0]["w_1"].shape[0]
    T = len(tokens)
    x = torch.from_numpy(w["tok_emb"][tokens].astype(np.float64) + w["pos_emb"][:T].astype(np.float64))[None]
    mask = torch.triu(torch.ones(T, T, dtype=torch.bool), diagonal=1)  # True = not allowed
    for L in w["layers"]:
        layer = torch.nn.TransformerEncoderLayer(H, nh, F, dropout=0.0, activation="gelu", norm_first=True,
                                                 batch_first=True, dtype=torch.float64)
        sd = {
            "self_attn.in_proj_weight": L["w_qkv"], "self_attn.in_proj_bias": L["b_qkv"],
            "self_attn.out_proj.weight": L["w_o"], "self_attn.out_proj.bias": L["b_o"],
            "linear1.weight": L["w_1"], "linear1.bias": L["b_1"], "linear2.weight": L["w_2"], "linear2.bias": L["b_2"],
            "norm1.weight": L["ln1_g"], "norm1.bias": L["ln1_b"], "norm2.weight": L["ln2_g"], "norm2.bias": L["ln2_b"],
        }
        layer.load_state_dict({k: torch.from_numpy(np.asarray(v, np.float64)) for k, v in sd.items()})
        layer.eval()
        with torch.no_grad():
            x = layer(x, src_mask=mask)
    y = torch.nn.functional.layer_norm(x[0, -1], (H,), torch.from_numpy(w["lnf_g"].astype(np.float64)),
                                       torch.from_numpy(w["lnf_b"].astype(np.float64)), eps=1e-5)
    logits = y @ torch.from_numpy(w["tok_emb"].astype(np.float64)).T
    return y.numpy(), logits.numpy()


def test_model_matches_torch_transformer_layer():
    w = tiny_weights(3)
    toks = [5, 17, 300, 2, 9, 511, 0, 44]
    store = KVStore(TINY.n_layers, TINY.hidden)
    r = model.iteration(w, TINY.n_heads, [BatchItem(0, toks, 0)], store)
    y, logits = torch_reference_prefill(w, TINY.n_heads, toks)
    np.testing.assert_allclose(r.hidden[0], y, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(r.logits[0], logits, rtol=1e-10, atol=1e-10)


# --------------------------------------------------------------------------- #
# selective batching == unbatched == padded+masked; K/V cache == recompute
# --------------------------------------------------------------------------- #
def build_contexts(w, prompts):
    """Prefill each prompt on its own; returns the store and the last tokens."""
    store = KVStore(TINY.n_layers, TINY.hidden)
    nxt = {}
    for rid, p in prompts.items():
        r = model.iteration(w, TINY.n_heads, [BatchItem(rid, p, 0)], store)
        nxt[rid] = r.next_tokens[0]
    return store, nxt


def mixed_tiny_batch(w):
    prompts = {10: [1, 2, 3, 4, 5], 11: [7], 12: [100, 200, 300, 400, 500, 6, 7, 8, 9, 10, 11]}
    store, nxt = build_contexts(w, prompts)
    batch = [BatchItem(10, [nxt[10]], 5), BatchItem(20, [3, 4], 0), BatchItem(11, [nxt[11]], 1),
             BatchItem(21, [9, 8, 7], 0), BatchItem(12, [nxt[12]], 11), BatchItem(22, [42], 0)]
    return store, batch


def test_selective_equals_unbatched_and_padded():
    w = tiny_weights(4)
    store, batch = mixed_tiny_batch(w)
    a = model.iteration(w, TINY.n_heads, batch, store.copy())
    b = unbatched.iteration(w, TINY.n_heads, batch, store.copy())
    c = padded.iteration(w, TINY.n_heads, batch, store.copy())
    for other in (b, c):
        np.testing.assert_allclose(a.hidden, other.hidden, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(a.logits, other.logits, rtol=1e-10, atol=1e-10)
        assert a.next_tokens == other.next_tokens


def test_kv_cache_equals_recompute():
    w = tiny_weights(5)
    seq = [3, 1, 4, 1, 5, 9, 2, 6]
    store = KVStore(TINY.n_layers, TINY.hidden)
    model.iteration(w, TINY.n_heads, [BatchItem(0, seq[:5], 0)], store)
    for p in range(5, len(seq)):
        inc = model.iteration(w, TINY.n_heads, [BatchItem(0, [seq[p]], p)], store)
        full = unbatched.recompute(w, TINY.n_heads, seq[:p + 1])
        np.testing.assert_allclose(inc.logits, full.logits, rtol=1e-10, atol=1e-10)


def test_flatten_case2_448():
    g = json.load(open(os.path.join(GOLD, "estelledc_case2_flatten.json")))
    H = 8
    rows = [np.zeros((L, H)) for L in g["prompt_lengths"]]
    assert model.flatten(rows).shape == (g["flattened_rows"], H)
    batch = [BatchItem(i, [0] * L, 0) for i, L in enumerate(g["prompt_lengths"])]
    assert model.offsets(batch) == [0, 128, 192, 448]


def test_flatten_houmin_7_rows():
    g = json.load(open(os.path.join(GOLD, "houmin_selective_batch.json")))
    H = 4
    x3, x4 = np.zeros((2, H)), np.zeros((3, H))
    assert model.flatten([x3, x4]).shape == (g["rows_x3_x4"], H)
    batch = [np.zeros((1, H)), np.zeros((1, H)), x3, x4]
    x = model.flatten(batch)
    assert x.shape == (g["rows_batch"], H)
    assert (x @ np.zeros((H, g["qkv_width_factor"] * H))).shape == (7, 3 * H)


def test_phase_mismatch_rejected():
    w = tiny_weights(6)
    store = KVStore(TINY.n_layers, TINY.hidden)
    with pytest.raises(ValueError):
        model.iteration(w, TINY.n_heads, [BatchItem(0, [1], 3)], store)


# --------------------------------------------------------------------------- #
# the pins catch plausible mistakes (mistakes planted in a copy of the oracle)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("mutation", ["no_scale", "swap_kv", "tanh_gelu", "unbiased_var", "post_ln"])
def test_pins_catch_planted_mistakes(mutation, monkeypatch):
    w = tiny_weights(3)
    toks = [5, 17, 300, 2, 9, 511, 0, 44]
    if mutation == "no_scale":
        orig = model.attention_one
        monkeypatch.setattr(model, "attention_one", lambda q, k, v, p, nh: orig(q * math.sqrt(q.shape[1] // nh), k, v, p, nh))
    elif mutation == "swap_kv":
        orig = model.attention_one
        monkeypatch.setattr(model, "attention_one", lambda q, k, v, p, nh: orig(q, v, k, p, nh))
    elif mutation == "tanh_gelu":
        monkeypatch.setattr(model, "gelu", lambda x: 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3))))
    elif mutation == "unbiased_var":
        def ln(x, g, b, eps=1e-5, dtype=np.float64):
            x = np.asarray(x, dtype)
            m = x.mean(-1, keepdims=True)
            return (x - m) / np.sqrt(x.var(-1, ddof=1, keepdims=True) + eps) * g + b
        monkeypatch.setattr(model, "layer_norm", ln)
    elif mutation == "post_ln":
        w = dict(w)
        w["layers"] = [dict(L, ln1_g=L["ln2_g"], ln2_g=L["ln1_g"]) for L in w["layers"]]
    store = KVStore(TINY.n_layers, TINY.hidden)
    r = model.iteration(w, TINY.n_heads, [BatchItem(0, toks, 0)], store)
    y, logits = torch_reference_prefill(tiny_weights(3), TINY.n_heads, toks)
    assert not np.allclose(r.logits[0], logits, rtol=1e-6, atol=1e-8)


def test_chunked_prompt_equals_whole_prompt():
    """A prompt processed in chunks (each chunk attending to the K/V the earlier
    chunks cached) gives the same last-row hidden state and logits as the whole
    prompt at once: the chunked-prefill schedule computes the same function."""
    w = tiny_weights(7)
    seq = [5, 17, 3, 250, 9, 1, 44, 8, 120, 6, 2, 77, 31]
    whole = model.iteration(w, TINY.n_heads, [BatchItem(0, seq, 0)], KVStore(TINY.n_layers, TINY.hidden))
    for cuts in ([4], [1, 7], [6, 11, 12]):
        store = KVStore(TINY.n_layers, TINY.hidden)
        bounds = [0] + cuts + [len(seq)]
        for a, b in zip(bounds, bounds[1:]):
            res = model.iteration(w, TINY.n_heads, [BatchItem(0, seq[a:b], a)], store)
        np.testing.assert_allclose(res.hidden, whole.hidden, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(res.logits, whole.logits, rtol=1e-10, atol=1e-10)
        assert res.next_tokens == whole.next_tokens


def test_float32_oracle_matches_float64():
    """The float32 form of the oracle (used only to time the CPU baseline in the
    precision the target names) computes the same iteration: within float32
    rounding of the float64 result, and the same greedy tokens."""
    w = tiny_weights(9)
    batch = [BatchItem(0, [5, 17, 300, 2], 0), BatchItem(1, [9, 511], 0)]
    r64 = model.iteration(w, TINY.n_heads, batch, KVStore(TINY.n_layers, TINY.hidden))
    r32 = model.iteration(w, TINY.n_heads, batch, KVStore(TINY.n_layers, TINY.hidden, np.float32), dtype=np.float32)
    assert r32.logits.dtype == np.float32 and r32.hidden.dtype == np.float32
    np.testing.assert_allclose(r32.hidden, r64.hidden, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(r32.logits, r64.logits, rtol=1e-4, atol=1e-4)
    assert r32.next_tokens == r64.next_tokens


def test_agreement_rule_rejects_clear_flips():
    """The GPU tests' agreement rule: at GPT-3 widths a disagreement is accepted
    only as a near-tie (oracle margin within a few RMS logit errors of the
    row) and only up to the bf16 flip floor; a flip with a clear margin, or
    too many flips, fails, and elsewhere 99 % is required."""
    from gpu_util import assert_agreement, disagreements
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((100, 5000))
    noise = 1e-3 * rng.standard_normal((100, 5000))
    gpu = ref + noise
    top2 = np.argsort(ref, 1)[:, -2:]
    near = int(np.argmin(ref[np.arange(100), top2[:, 1]] - ref[np.arange(100), top2[:, 0]]))
    gpu[near, top2[near, 0]] = gpu[near, top2[near, 1]] + 1e-6  # a near-tie flip
    got = gpu.argmax(1)
    tokens = ref.argmax(1).tolist()
    mm = disagreements(got, gpu, ref, tokens)
    assert len(mm) == 1 and mm[0]["row"] == near
    agree = 1 - len(mm) / 100
    if mm[0]["ref_margin"] <= 6 * mm[0]["row_rms_err"]:
        assert_agreement(agree, 100, mm, wide=True)
    with pytest.raises(AssertionError):  # one flip in 50 tokens is 98 %
        assert_agreement(1 - len(mm) / 50, 50, mm, wide=False)
    clear = gpu.copy()
    clear[3, int(np.argmin(ref[3]))] = ref[3].max() + 1.0  # the lowest logit pushed to the top: a bug
    mm2 = disagreements(clear.argmax(1), clear, ref, tokens)
    with pytest.raises(AssertionError):
        assert_agreement(1 - len(mm2) / 100, 100, mm2, wide=True)
    many = gpu.copy()  # five near-tie flips in 100 tokens: above the 3 % floor
    for r in np.argsort(ref[np.arange(100), top2[:, 1]] - ref[np.arange(100), top2[:, 0]])[:5]:
        many[r, top2[r, 0]] = many[r, top2[r, 1]] + 1e-6
    mm3 = disagreements(many.argmax(1), many, ref, tokens)
    assert len(mm3) == 5
    with pytest.raises(AssertionError):
        assert_agreement(0.95, 100, mm3, wide=True)
