"""The seeded input generators follow the stated input recipe (CPU, no GPU):
the workloads' shapes, N(0,1) activations and logits, tie-free logit rows,
the permutation order of the tiny workload, the skew of the Zipf(1.1) prior
on the 64-token decode batch, and the spread of the decoded expert weights.
Statistics use the CPU generator (the GPU one draws other numbers from the
same seeds), with margins far wider than their sampling error."""
import numpy as np
import torch

import oracle
import synth


def test_workload_shapes():
    W = synth.WORKLOADS
    big = (4096, 256, 2048, 8)  # d, E, f, k of the DeepSeek V4 Flash routed-expert layer
    for name, T, routing, down in [("decode1", 1, "normal", "mxfp4"), ("decode64", 64, "zipf", "mxfp4"),
                                   ("prefill", 4096, "normal", "mxfp4"), ("q2k", 2048, "normal", "q2k"),
                                   ("q2k_decode1", 1, "normal", "q2k"), ("q2k_decode64", 64, "zipf", "q2k")]:
        wl = W[name]
        assert (wl.T, wl.d, wl.E, wl.f, wl.k, wl.routing, wl.down) == (T, *big, routing, down), name
    # the reduced cases for profiler captures keep the tokens per expert of their full workloads
    for small, full in [("prefill_e32", "prefill"), ("q2k_e64", "q2k")]:
        s, f = W[small], W[full]
        assert s.T * s.k / s.E == f.T * f.k / f.E and (s.d, s.f, s.k) == (f.d, f.f, f.k)


def test_activations_are_standard_normal_in_bf16():
    wl = synth.WORKLOADS["decode64"]
    x = synth.make_x(wl)
    assert x.dtype == torch.bfloat16 and tuple(x.shape) == (64, 4096)
    v = x.float()
    assert abs(v.mean().item()) < 0.01 and abs(v.std().item() - 1.0) < 0.01
    assert torch.equal(synth.make_x(wl), x)  # seeded: the same bytes on every call


def test_logit_rows_are_tie_free_and_normal():
    for name in ("decode64", "prefill"):
        lg = synth.make_logits(synth.WORKLOADS[name])
        srt, _ = lg.sort(dim=1)
        assert not bool((srt[:, 1:] == srt[:, :-1]).any()), name
    lg = synth.make_logits(synth.WORKLOADS["prefill"])
    assert abs(lg.mean().item()) < 0.01 and abs(lg.std().item() - 1.0) < 0.01


def test_tie_breaking_touches_only_rows_with_ties():
    g = torch.Generator().manual_seed(5)
    lg = torch.tensor([[0.5, 0.5, -1.0, 2.0], [0.1, 0.2, 0.3, 0.4]])
    out = synth._break_ties(lg, g)
    assert torch.equal(out[1], lg[1])
    assert out[0, 0] != out[0, 1] and (out[0] - lg[0]).abs().max().item() <= 3 * 2.0 ** -20


def test_tiny_logits_follow_their_permutation():
    """tiny: randperm(E) * 0.5 + N(0, 0.01): the ranking is the permutation's."""
    wl = synth.WORKLOADS["tiny"]
    lg = synth.make_logits(wl).numpy()
    base = np.rint(lg / 0.5)
    assert np.abs(lg - 0.5 * base).max() < 0.1
    for row in base:
        assert sorted(row.astype(int).tolist()) == list(range(wl.E))


def test_zipf_prior_skews_the_decode_batch():
    """decode64: N(0,1) + log Zipf(1.1) prior concentrates 64 tokens x 8 slots
    on about 50 experts; plain N(0,1) logits spread them over about 220."""
    zipf, normal = [], []
    for seed in range(3):
        for routing, acc in (("zipf", zipf), ("normal", normal)):
            wl = synth.Workload("z", 64, 4096, 256, 2048, 8, seed, seed, routing)
            idx, _ = oracle.route(synth.make_logits(wl).numpy(), 8)
            cnt = np.bincount(idx.ravel(), minlength=256)
            acc.append((len(np.unique(idx)), np.sort(cnt)[-8:].sum() / cnt.sum()))
    for U, top8 in zipf:
        assert 30 <= U <= 90 and top8 > 0.4
    for U, top8 in normal:
        assert U >= 190 and top8 < 0.15


def test_prefill_batch_reaches_every_expert():
    idx, _ = oracle.route(synth.make_logits(synth.WORKLOADS["prefill"]).numpy(), 8)
    cnt = np.bincount(idx.ravel(), minlength=256)
    assert cnt.min() > 0 and abs(cnt.mean() - 128) < 1e-9  # 4096 x 8 / 256 tokens per expert on average


def test_decoded_weights_keep_the_generated_spread():
    """Weights are drawn N(0, 0.02) and stored in MXFP4 (gate/up, down) or
    Q2_K (down); decoded, they keep that spread to a few per cent."""
    for down in ("mxfp4", "q2k"):
        wl = synth.Workload("w_" + down, 2, 512, 2, 512, 1, 3, 3, "normal", down)
        W = {k: v.numpy() for k, v in synth.make_layer_weights(wl).items()}
        wg, wu, wd = oracle.dequant_expert({"d": wl.d, "E": wl.E, "f": wl.f}, W, 1)
        for m in (wg, wu, wd):
            assert abs(m.mean()) < 0.002 and abs(m.std() / 0.02 - 1.0) < 0.1, down
