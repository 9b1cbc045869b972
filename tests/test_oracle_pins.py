"""Pins of the fp64 oracle to things other than itself: library routines (torch
fp64 layer_norm, conv1d, glu, scaled-dot-product attention), closed forms, the
relShift cross-check, the streaming == offline invariant and the receptive-field
arithmetic the pages state."""
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from cache_aware_conformer_gb300 import synth
from cache_aware_conformer_gb300.config import TINY, DTYPE_F32
from oracle import conformer as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
T64 = torch.float64


def rng(seed=0):
    return np.random.default_rng(seed)


def tiny(**kw):
    return replace(TINY, **kw)


def weights(cfg, seed=0):
    return O.weights_f64(synth.make_weights(cfg, seed))


# ---------------------------------------------------------------------------
# elementary pieces against torch
# ---------------------------------------------------------------------------

def test_layer_norm_matches_torch():
    r = rng(1)
    x, g, b = r.normal(size=(7, 96)) * 3 + 1, r.normal(size=96), r.normal(size=96)
    ref = F.layer_norm(torch.tensor(x), (96,), torch.tensor(g), torch.tensor(b), eps=1e-5).numpy()
    np.testing.assert_allclose(O.layer_norm(x, g, b), ref, rtol=0, atol=1e-12)


def test_layer_norm_closed_form_zero_mean_unit_var():
    x = rng(2).normal(size=(5, 64)) * 7 - 3
    y = O.layer_norm(x, np.ones(64), np.zeros(64))
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    var = (y ** 2).mean(-1)
    np.testing.assert_allclose(var, x.var(-1) / (x.var(-1) + 1e-5), atol=1e-12)


@pytest.mark.parametrize("pad", [2, 0])
def test_conv_stage_matches_torch_conv1d(pad):
    r = rng(3)
    T, C, D = 31, 12, 10
    x, w, b = r.normal(size=(T, C)), r.normal(size=(D, 3, C)), r.normal(size=D)
    xt = torch.tensor(x.T[None])                                  # [1, C, T]
    wt = torch.tensor(np.transpose(w, (0, 2, 1)))                 # [D, C, 3]
    ref = F.relu(F.conv1d(F.pad(xt, (pad, 0)), wt, torch.tensor(b), stride=2))[0].numpy().T
    np.testing.assert_allclose(O.conv_stage(x, w, b, pad), ref, rtol=0, atol=1e-12)


def test_glu_matches_torch_and_zero_gate_halves():
    a = rng(4).normal(size=(6, 40))
    np.testing.assert_allclose(O.glu(a), F.glu(torch.tensor(a), dim=-1).numpy(), atol=1e-14)
    v = a[:, :20]
    np.testing.assert_array_equal(O.glu(np.concatenate([v, np.zeros_like(v)], 1)), 0.5 * v)


def test_feed_forward_matches_torch_composition():
    r = rng(5)
    D, FF = 16, 40
    W = {"ln_g": r.normal(size=D), "ln_b": r.normal(size=D), "w1": r.normal(size=(FF, D)),
         "b1": r.normal(size=FF), "w2": r.normal(size=(D, FF)), "b2": r.normal(size=D)}
    x = r.normal(size=(9, D))
    t = {k: torch.tensor(v) for k, v in W.items()}
    xt = torch.tensor(x)
    h = F.silu(F.linear(F.layer_norm(xt, (D,), t["ln_g"], t["ln_b"], eps=1e-5), t["w1"], t["b1"]))
    ref = (xt + 0.5 * F.linear(h, t["w2"], t["b2"])).numpy()
    np.testing.assert_allclose(O.feed_forward(x, W, ""), ref, atol=1e-12)


def _conv_weights(r, D, K=9):
    return {"ln_g": r.normal(size=D), "ln_b": r.normal(size=D),
            "w_pw1": r.normal(size=(2 * D, D)) / 4, "b_pw1": r.normal(size=2 * D),
            "w_dw": r.normal(size=(D, K)), "b_dw": r.normal(size=D),
            "bn_g": r.normal(size=D), "bn_b": r.normal(size=D),
            "w_pw2": r.normal(size=(D, D)) / 4, "b_pw2": r.normal(size=D)}


def test_conv_module_matches_torch_composition():
    r = rng(6)
    D, T = 12, 23
    W = _conv_weights(r, D)
    x = r.normal(size=(T, D))
    out, full, _ = O.conv_module(x, W, "", np.zeros((8, D)))
    t = {k: torch.tensor(v) for k, v in W.items()}
    xt = torch.tensor(x)
    g = F.glu(F.linear(F.layer_norm(xt, (D,), t["ln_g"], t["ln_b"], eps=1e-5), t["w_pw1"], t["b_pw1"]), dim=-1)
    dw = F.conv1d(F.pad(g.T[None], (8, 0)), t["w_dw"][:, None, :], t["b_dw"], groups=D)[0].T
    ref = xt + F.linear(F.silu(t["bn_g"] * dw + t["bn_b"]), t["w_pw2"], t["b_pw2"])
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-11)
    assert full.shape == (8 + T, D)


def test_depthwise_delta_kernel_is_a_shift():
    r = rng(7)
    D, T = 8, 15
    W = _conv_weights(r, D)
    for k0 in (0, 4, 8):
        W["w_dw"] = np.zeros((D, 9))
        W["w_dw"][:, k0] = 1.0
        W["b_dw"], W["bn_g"], W["bn_b"] = np.zeros(D), np.ones(D), np.zeros(D)
        prev = r.normal(size=(8, D))
        _, full, (g, y) = O.conv_module(r.normal(size=(T, D)), W, "", prev)
        # output t reads glu_{t-8+k0}: index t + k0 of [prev | glu_new]
        np.testing.assert_array_equal(y, O.silu(full[k0: k0 + T]))


def test_sinusoid_closed_forms():
    r = np.array([-5, -1, 0, 1, 3, 77])
    pe = O.sinusoid(r, 16)
    np.testing.assert_allclose(pe[:, 0], np.sin(r), atol=1e-15)
    np.testing.assert_allclose(pe[:, 1], np.cos(r), atol=1e-15)
    np.testing.assert_allclose(pe[:, 14], np.sin(r * 10000.0 ** (-14 / 16)), atol=1e-15)
    np.testing.assert_allclose(pe[:, 0::2] ** 2 + pe[:, 1::2] ** 2, 1.0, atol=1e-14)
    np.testing.assert_array_equal(pe[2], np.tile([0.0, 1.0], 8))


# ---------------------------------------------------------------------------
# attention: SDPA special cases, relShift cross-check
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, bias):
    return F.scaled_dot_product_attention(torch.tensor(q)[None], torch.tensor(k)[None],
                                          torch.tensor(v)[None], attn_mask=torch.tensor(bias)[None])[0].numpy()


def test_attention_reduces_to_textbook_softmax_attention():
    """pbu = pbv = 0, W_pos = 0 and an all-visible mask: plain multi-head attention."""
    r = rng(8)
    T, D, H = 11, 24, 3
    hd = D // H
    q, k, v = (r.normal(size=(T, D)) for _ in range(3))
    pos = np.arange(T)
    out = O.rel_pos_attention(q, k, v, pos, pos, np.zeros((D, D)), np.zeros((H, hd)), np.zeros((H, hd)),
                              H, O.chunk_mask(pos, pos, chunk=T, left=T))
    for h in range(H):
        sl = slice(h * hd, (h + 1) * hd)
        np.testing.assert_allclose(out[:, sl], _sdpa(q[:, sl], k[:, sl], v[:, sl], np.zeros((T, T))), atol=1e-12)


def test_chunk_mask_matches_chunk_index_construction():
    """Mask on absolute positions == the same rule stated on chunk indices
    (left context 70 frames = 35 chunks of 2), keys before the start absent."""
    pq = np.arange(200, 260)
    pk = np.arange(100, 262)
    m = O.chunk_mask(pq, pk, 2, 70)
    cq, ck = (pq // 2)[:, None], (pk // 2)[None, :]
    ref = (ck <= cq) & (ck >= cq - 35) & (pk[None, :] >= 0)
    np.testing.assert_array_equal(m, ref)
    # every query sees itself, never a key beyond its chunk end, and at most 72 keys
    assert m[np.arange(60), np.arange(60) + 100].all()
    assert m.sum(1).max() == 72


def test_rel_shift_equals_direct_rel_indexing():
    r = rng(9)
    T, hd = 9, 8
    qv = r.normal(size=(T, hd))
    wrow = r.normal(size=(hd, 16))
    rows = lambda rv: O.sinusoid(rv, 16) @ wrow.T
    shifted = O.bd_term_rel_shift(qv, rows)
    i, j = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    direct = np.einsum("td,tjd->tj", qv, rows((i - j).reshape(-1)).reshape(T, T, hd))
    np.testing.assert_allclose(shifted, direct, atol=1e-12)


def test_rel_pos_attention_matches_relshift_plus_sdpa():
    """Whole rel-pos attention (content + position term, chunked mask, softmax,
    probs@V) against torch SDPA whose additive bias is the relShift bd term."""
    r = rng(10)
    T, D, H = 13, 32, 4
    hd = D // H
    q, k, v = (r.normal(size=(T, D)) for _ in range(3))
    wpos = r.normal(size=(D, D)) / 5
    pbu, pbv = r.normal(size=(H, hd)) * 0.3, r.normal(size=(H, hd)) * 0.3
    pos = np.arange(T)
    mask = O.chunk_mask(pos, pos, chunk=2, left=4)
    out = O.rel_pos_attention(q, k, v, pos, pos, wpos, pbu, pbv, H, mask)
    for h in range(H):
        sl = slice(h * hd, (h + 1) * hd)
        rows = lambda rv: (O.sinusoid(rv, D) @ wpos.T)[:, sl]
        bd = O.bd_term_rel_shift(q[:, sl] + pbv[h], rows) / math.sqrt(hd)
        bias = np.where(mask, bd, -np.inf)
        ref = _sdpa(q[:, sl] + pbu[h], k[:, sl], v[:, sl], bias)
        np.testing.assert_allclose(out[:, sl], ref, atol=1e-12)


# ---------------------------------------------------------------------------
# lengths and receptive field
# ---------------------------------------------------------------------------

def test_offline_encoder_matches_torch_composition():
    """The whole offline encode against the same network written with torch
    primitives: subsampling (three causal stride-2 conv1d + ReLU, then the
    linear), every layer as FF1 (half residual) -> attention -> conv module ->
    FF2 (half residual) -> ln_out, then the joint projection.  Attention is
    textbook multi-head softmax attention here (position terms zero, a context
    and chunk covering the sequence), so any slip in module order, residual
    weight, LayerNorm placement or a weight's role fails."""
    cfg = tiny(att_left=1000, att_chunk=64)
    W = weights(cfg, 3)
    for l in range(cfg.n_layers):
        for n in ("wpos", "pbu", "pbv"):
            W[f"l{l}.att.{n}"] = np.zeros_like(W[f"l{l}.att.{n}"])
    mel = synth.make_mel(200, 5)                                   # 25 frames, all in one chunk
    enc, joint = O.encode_offline(mel, W, cfg)
    t = {k: torch.tensor(v) for k, v in W.items()}
    D, H, kk = cfg.d_model, cfg.n_heads, cfg.dw_kernel
    hd = D // H
    y = torch.tensor(mel, dtype=T64)
    for st in (1, 2, 3):                                            # weights stored [out][tap][in]
        y = F.relu(F.conv1d(F.pad(y.T[None], (2, 0)), t[f"sub.w{st}"].permute(0, 2, 1), t[f"sub.b{st}"],
                            stride=2)[0].T)
    x = F.linear(y, t["sub.wo"], t["sub.bo"])

    def ln(v, p):
        return F.layer_norm(v, (D,), t[p + "ln_g"], t[p + "ln_b"], eps=1e-5)

    def ff(v, p):
        return v + 0.5 * F.linear(F.silu(F.linear(ln(v, p), t[p + "w1"], t[p + "b1"])), t[p + "w2"], t[p + "b2"])

    for l in range(cfg.n_layers):
        p = f"l{l}."
        x = ff(x, p + "ff1.")
        a = ln(x, p + "att.")
        q, k, v = (F.linear(a, t[p + f"att.w{c}"], t[p + f"att.b{c}"]).view(-1, H, hd).transpose(0, 1)
                   for c in "qkv")
        o = F.scaled_dot_product_attention(q[None], k[None], v[None])[0].transpose(0, 1).reshape(-1, D)
        x = x + F.linear(o, t[p + "att.wo"], t[p + "att.bo"])
        g = F.glu(F.linear(ln(x, p + "conv."), t[p + "conv.w_pw1"], t[p + "conv.b_pw1"]), dim=-1)
        dw = F.conv1d(F.pad(g.T[None], (kk - 1, 0)), t[p + "conv.w_dw"][:, None, :], t[p + "conv.b_dw"],
                      groups=D)[0].T
        x = x + F.linear(F.silu(t[p + "conv.bn_g"] * dw + t[p + "conv.bn_b"]), t[p + "conv.w_pw2"],
                         t[p + "conv.b_pw2"])
        x = ff(x, p + "ff2.")
        x = ln(x, p + "out.")
    assert enc.shape == (25, D)
    np.testing.assert_allclose(enc, x.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(joint, F.linear(x, t["joint.w"], t["joint.b"]).numpy(), rtol=0, atol=1e-10)


def test_length_arithmetic():
    fw = GOLDEN["offline_window"]
    assert O.subsampled_len(fw["mel"]) == fw["frames"]
    assert O.subsampled_len(320) == 40 and O.subsampled_len(3000) == 375 and O.subsampled_len(6000) == 750
    cfg = tiny(d_model=8, n_heads=2, ff_dim=16, n_layers=1)
    W = weights(cfg)
    assert O.subsample(np.zeros((fw["mel"], 128)), W, 2).shape == (fw["frames"], 8)


def test_mel_tail_receptive_field_is_14_frames():
    """Perturbing mel frame t changes exactly the subsampled frames m with
    8m - 14 <= t <= 8m (bit-identical elsewhere)."""
    assert O.MEL_TAIL == GOLDEN["mel_tail_frames"]["value"]
    cfg = tiny(d_model=16, n_heads=2, ff_dim=32, n_layers=1)
    W = weights(cfg)
    mel = rng(11).normal(size=(200, 128))
    base = O.subsample(mel, W, 2)
    for t in (0, 7, 8, 50, 101, 199):
        m2 = mel.copy()
        m2[t] += 3.0
        changed = np.nonzero(np.any(O.subsample(m2, W, 2) != base, axis=1))[0]
        expect = [m for m in range(base.shape[0]) if 8 * m - 14 <= t <= 8 * m]
        # exactly the 14-frame field (frame 199 feeds no output of a 200-frame window)
        assert list(changed) == expect


def test_chunked_causality_of_the_layer_stack():
    """Perturbing subsampled frame p leaves every output at positions < floor(p/2)*2
    bit-identical, and changes the output at p itself."""
    cfg = tiny(att_left=6)
    W = weights(cfg)
    x0 = rng(12).normal(size=(30, cfg.d_model))

    def run(x):
        D = cfg.d_model
        for l in range(cfg.n_layers):
            x, _, _, _ = O.layer_step(x, W, l, cfg, np.zeros((0, D)), np.zeros((0, D)), np.zeros((8, D)), 0)
        return x

    base = run(x0)
    for p in (0, 5, 12, 29):
        x = x0.copy()
        x[p] += rng(p).normal(size=cfg.d_model)   # not a constant shift: LayerNorm removes those
        y = run(x)
        c = (p // 2) * 2
        np.testing.assert_array_equal(y[:c], base[:c])
        assert np.abs(y[p] - base[p]).max() > 1e-6


# ---------------------------------------------------------------------------
# streaming == offline (the pages' gate, in fp64)
# ---------------------------------------------------------------------------

def _stream(cfg, W, mel, sizes):
    enc = StreamRun(cfg, W)
    outs, i, k = [], 0, 0
    while i + 16 <= mel.shape[0]:
        n = min(sizes[k % len(sizes)], (mel.shape[0] - i) // 16 * 16)
        outs.append(enc.push(mel[i:i + n]))
        i += n
        k += 1
        assert enc.s.Lc == min(enc.s.subT, cfg.att_left)
        assert enc.s.mel_tail.shape[0] == 14
    outs.append(enc.flush(mel[i:]))
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])


class StreamRun:
    def __init__(self, cfg, W):
        self.s = O.StreamingEncoder(W, cfg)

    def push(self, m):
        return self.s.push(m)

    def flush(self, m):
        return self.s.flush(m)


@pytest.mark.parametrize("att_left,sizes,t_mel", [
    (70, [16], 320),            # config 1: 3.2 s, 160 ms pushes
    (70, [16, 32, 64], 1013),   # cache fills past 70 rows; ragged flush of 5 mel frames
    (6, [16], 203),             # short left context: cache trimming every push
    (6, [64, 16, 48], 400),     # pushes of n = 8, 2, 6 frames
])
def test_streaming_equals_offline(att_left, sizes, t_mel):
    cfg = tiny(att_left=att_left)
    W = weights(cfg)
    mel = synth.make_mel(t_mel, 3)
    enc_off, joint_off = O.encode_offline(mel, W, cfg)
    enc_st, joint_st = _stream(cfg, W, mel, sizes)
    assert enc_st.shape == enc_off.shape == (O.subsampled_len(t_mel), cfg.d_model)
    assert np.abs(enc_st - enc_off).max() <= 1e-9
    assert np.abs(joint_st - joint_off).max() <= 1e-9


def test_streaming_after_reset_equals_offline_of_new_utterance():
    cfg = tiny(att_left=10)
    W = weights(cfg)
    s = O.StreamingEncoder(W, cfg)
    pre = synth.make_mel(96, 4)
    for i in range(0, 96, 16):
        s.push(pre[i:i + 16])
    s.reset()
    mel = synth.make_mel(160, 5)
    outs = [s.push(mel[i:i + 16])[0] for i in range(0, 160, 16)]
    off, _ = O.encode_offline(mel, W, cfg)
    assert np.abs(np.concatenate(outs) - off).max() <= 1e-9


def test_cache_bytes_example_from_the_page():
    g = GOLDEN["kv_cache_bytes_example"]
    assert g["rows"] * g["width"] * g["bytes_per_value"] * g["kv"] * g["layers"] == g["value"]


# ---------------------------------------------------------------------------
# provisional tail
# ---------------------------------------------------------------------------

def _prov(cfg, W, mel, push=32):
    s = O.ProvisionalTailEncoder(W, cfg)
    outs = []
    i = 0
    while i + push <= mel.shape[0]:
        outs.append(s.push(mel[i:i + push])[0])
        i += push
    outs.append(s.flush(mel[i:])[0])
    return np.concatenate(outs)


def test_provisional_tail_right_context_zero_is_exact():
    """With right context 0 the oracle takes the chunked mask (chunk 1 here), whose
    window [p-left, p] needs no lookahead, so the provisional-tail schedule must
    equal offline exactly.  (window_mask itself is pinned by the receptive-field
    test below and by its equality with chunk_mask at chunk 1.)"""
    cfg = tiny(right_context=0, att_chunk=1, emit_frames=4, lookahead_frames=16, att_left=10)
    W = weights(cfg)
    mel = synth.make_mel(483, 6)
    off, _ = O.encode_offline(mel, W, cfg)
    assert np.abs(_prov(cfg, W, mel) - off).max() <= 1e-9


def test_provisional_tail_with_unbounded_lookahead_is_exact():
    cfg = tiny(right_context=3, emit_frames=4, lookahead_frames=64, att_left=10)
    W = weights(cfg)
    mel = synth.make_mel(400, 7)              # 50 frames < 4 + 64: everything happens at flush
    off, _ = O.encode_offline(mel, W, cfg)
    assert np.abs(_prov(cfg, W, mel) - off).max() <= 1e-9


def test_provisional_tail_bounded_lookahead_drift_shrinks_with_lookahead():
    cfg = tiny(right_context=3, emit_frames=4, att_left=10)
    W = weights(cfg)
    mel = synth.make_mel(640, 8)
    off, _ = O.encode_offline(mel, W, cfg)
    d = [np.abs(_prov(replace(cfg, lookahead_frames=B), W, mel) - off).max() for B in (4, 8, 16)]
    assert d[0] > 0 and d[2] < d[0]


# ---------------------------------------------------------------------------
# right-context window mask ("True streaming encode", §Status: the Nemotron
# variant with right context 3, whose lookahead cascades through the layers)
# ---------------------------------------------------------------------------

def test_window_mask_with_no_right_context_is_chunk_mask_of_chunk_one():
    pq = np.arange(0, 90)
    pk = np.arange(-5, 95)
    for left in (0, 6, 70):
        np.testing.assert_array_equal(O.window_mask(pq, pk, left, 0), O.chunk_mask(pq, pk, 1, left))


def test_window_mask_receptive_field_of_one_layer():
    """One layer with right context 3 and left context 6 through layer_step and the
    window mask: perturbing frame p changes the attention output exactly at
    queries q in [p - 3, p + 6] (q sees keys [q - 6, q + 3]); the causal k = 9
    depthwise conv after it then reaches 8 frames further right, so the layer
    output changes exactly at [p - 3, p + 14] and is bit-identical elsewhere.
    An off-by-one at either edge of the mask moves one end of that set."""
    cfg = tiny(right_context=3, att_left=6, n_layers=1)
    W = weights(cfg)
    D = cfg.d_model
    x0 = rng(40).normal(size=(48, D))

    def run(x):
        tr = {}
        y, _, _, _ = O.layer_step(x, W, 0, cfg, np.zeros((0, D)), np.zeros((0, D)), np.zeros((8, D)), 0, tr)
        return y, tr["att"][0]

    base, base_att = run(x0)
    for p in (3, 10, 20, 33):
        x = x0.copy()
        x[p] += rng(p).normal(size=D)   # not a constant shift: LayerNorm removes those
        y, att = run(x)
        att_changed = np.nonzero(np.any(att != base_att, axis=1))[0]
        assert list(att_changed) == [q for q in range(48) if p - 3 <= q <= p + 6], p
        changed = np.nonzero(np.any(y != base, axis=1))[0]
        assert list(changed) == [q for q in range(48) if p - 3 <= q <= p + 14], p


def test_window_mask_edges_on_absolute_positions():
    """Keys before the stream start are absent; a query at p sees exactly the
    keys p - left .. p + right that exist."""
    pq = np.array([0, 1, 5, 40])
    pk = np.arange(-3, 60)
    m = O.window_mask(pq, pk, 6, 3)
    for i, p in enumerate(pq):
        assert list(pk[m[i]]) == [k for k in range(max(0, p - 6), p + 4)]
