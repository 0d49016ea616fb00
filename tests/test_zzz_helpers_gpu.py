"""The tensor helpers of the global scheduler, the pruning, the confidence head
and the DART tree on the GPU, against the oracle on small seeded cases (the
raw C calls behind them are covered case by case in
test_gpu_tree_markov_schedule.py)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _cuda(a, dt):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a).astype(dt))).cuda()


def _bf16(logits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(logits.raw.view(np.int16))).cuda().view(torch.bfloat16)


def test_schedule_global_and_prune_helpers():
    import lossless_draft_verification_gb300 as specv
    conf = synth.confidences(501, 40, 7)
    stale = synth.confidences(502, 40, 7)
    sps = synth.sps_table(4096)
    c, cs, t = _cuda(conf, np.float32), _cuda(stale, np.float32), _cuda(sps, np.float64)
    ell, theta = specv.schedule_global(c, t, conf_stale=cs)
    ref = oracle.schedule_global(conf, sps, conf_stale=stale)
    assert (ell.cpu().numpy() == ref.lengths).all()
    assert float(theta.cpu().numpy()[0]) == ref.theta_best
    lens = specv.prune_threshold(c, 0.5)
    assert (lens.cpu().numpy() == oracle.prune_threshold(conf, 0.5)).all()


def test_confidence_head_helper():
    """float32 accumulation of H + rank exact products, as in the raw-call test."""
    import lossless_draft_verification_gb300 as specv
    R, gamma, H, V, rank = 8, 7, 256, 1000, 64
    h = synth.make_logits(synth.normal(503, 1, (R, gamma, H)), "bf16")
    W1 = synth.make_logits(0.02 * synth.normal(503, 2, (V, rank)), "bf16")
    w = (synth.normal(503, 3, (H + rank,)) / np.sqrt(H + rank)).astype(np.float32)
    anchor = (synth.uniform_u24(503, 4, (R,)) * V).astype(np.int32)
    toks = (synth.uniform_u24(503, 5, (R, gamma)) * V).astype(np.int32)
    c = specv.confidence_head(_bf16(h), _bf16(W1), _cuda(w, np.float32), 0.5, _cuda(anchor, np.int32),
                              _cuda(toks, np.int32)).cpu().numpy()
    ref = oracle.confidence_head(h.f64, W1.f64, w, 0.5, anchor, toks)
    prev = np.concatenate([anchor[:, None], toks[:, :gamma - 1]], axis=1)
    mag = np.abs(h.f64) @ np.abs(w[:H].astype(np.float64)) + np.abs(W1.f64[prev]) @ np.abs(w[H:].astype(np.float64))
    assert (np.abs(c - ref) <= 1e-6 + (H + rank) * 2.0 ** -24 * mag / 4).all()


def test_dart_tree_helper():
    import lossless_draft_verification_gb300 as specv
    R, d, V, k, w, theta = 2, 4, 4096, 8, 4, 20
    logits = synth.make_logits(3.0 * synth.normal(504, 1, (R, d, V)), "bf16")
    par, tok, nn = specv.dart_tree(_bf16(logits), 1.0, k=k, w=w, theta=theta)
    ref = oracle.dart_tree(logits.f64, 1.0, k=k, w=w, theta=theta)
    assert (nn.cpu().numpy() == ref.n_nodes).all()
    assert (par.cpu().numpy() == ref.parents).all()
    assert (tok.cpu().numpy() == ref.tokens).all()
