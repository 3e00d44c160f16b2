"""Pins for the CPU oracle: hand-worked values, closed forms, library routines
and brute force, so that the oracle is checked against something other than
itself before it is used to check the CUDA library.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats.json")))


def _bits(x_bf16: torch.Tensor) -> np.ndarray:
    return x_bf16.contiguous().view(torch.int16).numpy().view(np.uint16)


def _dims(d, E, f, k):
    return {"d": d, "E": E, "f": f, "k": k}


def _const_layer(d, f, E, gate_byte, up_byte, down_byte, scale=127):
    return {
        "gate_codes": np.full((E, f, d // 2), gate_byte, np.uint8),
        "gate_scales": np.full((E, f, d // 32), scale, np.uint8),
        "up_codes": np.full((E, f, d // 2), up_byte, np.uint8),
        "up_scales": np.full((E, f, d // 32), scale, np.uint8),
        "down_codes": np.full((E, d, f // 2), down_byte, np.uint8),
        "down_scales": np.full((E, d, f // 32), scale, np.uint8),
    }


def _np_weights(W: dict) -> dict:
    return {k: v.cpu().numpy() for k, v in W.items()}


# ----------------------------------------------------------------- formats
def test_e2m1_table(oracle_lib):
    g = GOLDEN["e2m1_table"]
    for c, v in zip(g["codes"], g["values"]):
        got = oracle_lib.e2m1(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (c, got, v)


def test_e8m0(oracle_lib):
    g = GOLDEN["e8m0"]
    for b, v in zip(g["bytes"], g["values"]):
        assert oracle_lib.e8m0(b) == v
    assert math.isnan(oracle_lib.e8m0(255))


def test_mxfp4_block_nibble_order(oracle_lib):
    g = GOLDEN["mxfp4_block"]
    W = _const_layer(32, 32, 1, 0, 0, 0)
    W["gate_codes"][0, 0, 0] = g["code_byte"]
    W["gate_scales"][0, 0, 0] = g["scale_byte"]
    wg, _, _ = oracle_lib.dequant_expert(_dims(32, 1, 32, 1), W, 0)
    assert list(wg[0, :2]) == g["values"]
    assert np.all(wg[0, 2:] == 0) and np.all(wg[1:] == 0)


def test_mxfp4_scale_block_index(oracle_lib):
    # codes 0x22 = (1.0, 1.0); row 0 has scale 2^0 on block 0, 2^1 on block 1
    W = _const_layer(64, 32, 1, 0x22, 0x22, 0x22)
    W["gate_scales"][0, 0, 1] = 128
    W["down_scales"][0, 5, 0] = 126
    wg, wu, wd = oracle_lib.dequant_expert(_dims(64, 1, 32, 1), W, 0)
    assert np.all(wg[0, :32] == 1.0) and np.all(wg[0, 32:] == 2.0)
    assert np.all(wg[1:] == 1.0) and np.all(wu == 1.0)
    assert np.all(wd[5] == 0.5) and np.all(np.delete(wd, 5, axis=0) == 1.0)


def test_mxfp4_generator_hand_example(oracle_lib):
    g = GOLDEN["mxfp4_encoder"]
    w = torch.zeros(1, 32, dtype=torch.float32)
    w[0, :2] = torch.tensor(g["block_head"])
    codes, scales = synth.encode_mxfp4(w)
    assert int(scales[0, 0]) == g["scale_byte"]
    v = [oracle_lib.e2m1(int(codes[0, 0]) & 15) * oracle_lib.e8m0(int(scales[0, 0])),
         oracle_lib.e2m1(int(codes[0, 0]) >> 4) * oracle_lib.e8m0(int(scales[0, 0]))]
    assert v == g["values"]


def test_mxfp4_generator_error_bound(oracle_lib):
    """Each decoded weight is the nearest E2M1 grid point of w/2^s (within
    half a grid step), except above 6 where it saturates."""
    torch.manual_seed(0)
    w = torch.randn(8, 256) * 0.02
    codes, scales = synth.encode_mxfp4(w)
    grid = np.array(synth.E2M1_GRID)
    for r in range(8):
        for c in range(256):
            byte = int(codes[r, c // 2])
            code = byte & 15 if c % 2 == 0 else byte >> 4
            sc = oracle_lib.e8m0(int(scales[r, c // 32]))
            dec = oracle_lib.e2m1(code) * sc
            a = abs(float(w[r, c])) / sc
            nearest = grid[np.argmin(np.abs(grid - min(a, 6.0)))]
            assert abs(abs(dec) / sc - nearest) <= 1e-12 or abs(abs(a - nearest) - abs(a - abs(dec) / sc)) < 1e-12
            assert dec == 0 or math.copysign(1, dec) == math.copysign(1, float(w[r, c]))
        # the block rule: 6*2^s <= amax < 12*2^s
        for b in range(8):
            amax = float(w[r, 32 * b:32 * b + 32].abs().max())
            sc = oracle_lib.e8m0(int(scales[r, b]))
            assert 6 * sc <= amax < 12 * sc


def test_e4m3_golden(oracle_lib):
    g = GOLDEN["e4m3"]
    for v, b, dv in zip(g["values"], g["bytes"], g["decoded"]):
        assert oracle_lib.e4m3_encode(v) == b
        assert oracle_lib.e4m3_decode(b) == dv


def test_e4m3_against_torch(oracle_lib):
    # decode: every byte against torch's float8_e4m3fn
    allb = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        ref = float(allb[b])
        got = oracle_lib.e4m3_decode(b)
        assert (math.isnan(ref) and math.isnan(got)) or ref == got, b
    # encode: in-range values (torch's cast does not saturate, so stay below 448)
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-447, 447, 3000), rng.uniform(-0.03, 0.03, 3000),
                           np.ldexp(rng.integers(-1000, 1000, 500), -10)])
    ref = torch.tensor(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        got = oracle_lib.e4m3_encode(float(v))
        if v == 0 or (abs(v) < 2 ** -10 and got & 0x7F == 0):
            assert got & 0x7F == 0 and r & 0x7F == 0
        else:
            assert got == r, (v, got, r)
    # saturation
    assert oracle_lib.e4m3_encode(1e6) == 0x7E and oracle_lib.e4m3_encode(-500.0) == 0xFE


def test_mxfp8_block_golden(oracle_lib):
    g = GOLDEN["mxfp8_block"]
    v = np.zeros(32)
    v[:2] = g["block_head"]
    codes, scales = oracle_lib.mxfp8(v)
    assert int(scales[0]) == g["scale_byte"]
    dec = [oracle_lib.e4m3_decode(int(c)) * oracle_lib.e8m0(int(scales[0])) for c in codes[:2]]
    assert dec == g["decoded"]
    # all-zero block -> scale byte 127, codes 0
    codes, scales = oracle_lib.mxfp8(np.zeros(32))
    assert int(scales[0]) == 127 and not codes.any()


def test_q2k_golden(oracle_lib):
    g = GOLDEN["q2k"]
    blk = np.zeros(84, np.uint8)
    blk[0] = g["scale_byte"]
    q = g["q"]
    blk[16] = q[0] | (q[1] << 2) | (q[2] << 4) | (q[3] << 6)
    blk[80:82] = np.array([g["d_bits"]], np.uint16).view(np.uint8)
    blk[82:84] = np.array([g["dmin_bits"]], np.uint16).view(np.uint8)
    got = [oracle_lib.q2k_weight(blk, i) for i in range(4)]
    assert got == g["values"]
    # sub-block index: weight 16 uses scale byte 1 (sc=1, m=1): 0.5*1*q - 0.25*1
    blk[1] = 0x11
    blk[16 + 4] = 3  # weight 16, q = 3
    assert oracle_lib.q2k_weight(blk, 16) == 0.5 * 3 - 0.25
    assert oracle_lib.q2k_weight(blk, 17) == -0.25
    assert oracle_lib.q2k_weight(blk, 15) == -1.0  # still sub-block 0, q = 0


def test_q2k_generator_bound(oracle_lib):
    torch.manual_seed(3)
    w = torch.randn(4, 512) * 0.02
    blocks = synth.encode_q2k(w).numpy()
    for r in range(4):
        for sb in range(2):
            blk = blocks[r, sb]
            d = oracle_lib.half(int(blk[80]) | (int(blk[81]) << 8))
            for i in range(256):
                sc = blk[i // 16] & 15
                dec = oracle_lib.q2k_weight(blk, i)
                # within one quantisation step of the source value
                assert abs(dec - float(w[r, 256 * sb + i])) <= d * sc * 0.5 + 0.02 * 0.05


# ----------------------------------------------------------------- routing
def test_softmax_two(oracle_lib):
    g = GOLDEN["softmax2"]
    idx, w = oracle_lib.route(np.array([[g["logits"][0], g["logits"][1], -5.0]], np.float32), 2)
    assert list(idx[0]) == [0, 1]
    assert abs(w[0, 0] - g["weights"][0]) < 1e-15 and abs(w[0, 1] - g["weights"][1]) < 1e-15


def test_route_signed_zero_and_nan(oracle_lib):
    """The reading of the pages' routing at its edges: -0 ranks with +0 (a tie,
    broken by the lower index) and NaN ranks with -inf; worked by hand."""
    nan, inf = float("nan"), float("inf")
    logits = np.array([[-0.0, 0.0, nan, -inf, 1.0]], np.float32)
    idx, w = oracle_lib.route(logits, 5)
    assert idx.tolist() == [[4, 0, 1, 2, 3]]
    e1 = math.exp(-1.0)
    z = 1.0 + 2 * e1
    assert np.allclose(w[0], [1.0 / z, e1 / z, e1 / z, 0.0, 0.0], rtol=0, atol=1e-15)
    idx3, w3 = oracle_lib.route(logits, 3)
    assert idx3.tolist() == [[4, 0, 1]]
    assert abs(w3.sum() - 1.0) < 1e-15


def test_topk_brute_force_with_ties(oracle_lib):
    rng = np.random.default_rng(5)
    T, E, k = 50, 37, 6
    logits = rng.integers(-4, 5, size=(T, E)).astype(np.float32)  # many exact ties
    logits[::3] = rng.standard_normal((len(logits[::3]), E)).astype(np.float32)
    idx, w = oracle_lib.route(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(idx[t]) == order
        z = sum(math.exp(float(logits[t, e]) - float(logits[t, order[0]])) for e in order)
        for j, e in enumerate(order):
            assert abs(w[t, j] - math.exp(float(logits[t, e]) - float(logits[t, order[0]])) / z) < 1e-14
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_group_is_stable_sort(oracle_lib):
    rng = np.random.default_rng(7)
    T, E, k = 300, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle_lib.route(logits, k)
    G = oracle_lib.group(idx, E)
    pairs = sorted(((int(idx[t, j]), t, j) for t in range(T) for j in range(k)))
    assert list(G["perm_tok"]) == [p[1] for p in pairs]
    assert list(G["perm_slot"]) == [p[2] for p in pairs]
    assert G["offsets"][0] == 0 and G["offsets"][E] == T * k
    assert list(np.diff(G["offsets"])) == list(G["counts"])
    assert list(G["counts"]) == [int((idx == e).sum()) for e in range(E)]
    for t in range(T):
        assert (G["perm_tok"] == t).sum() == k
        for j in range(k):
            p = G["inv"][t, j]
            assert G["perm_tok"][p] == t and G["perm_slot"][p] == j


# ----------------------------------------------------------------- layer
def test_closed_form_single_expert(oracle_lib):
    d = f = 32
    W = _const_layer(d, f, 1, 0x22, 0x11, 0x22)  # gate 1.0, up 0.5, down 1.0
    x = torch.ones(1, d, dtype=torch.bfloat16)
    idx, w = np.zeros((1, 1), np.int32), np.ones((1, 1))
    out = oracle_lib.forward(_dims(d, 1, f, 1), W, _bits(x), idx, w, [0])
    g, u = 32.0, 16.0
    h = g / (1.0 + math.exp(-g)) * u
    assert np.allclose(out[0], 32 * h, rtol=1e-15, atol=0)


def test_combine_weights_follow_slots(oracle_lib):
    d = f = 32
    W = _const_layer(d, f, 2, 0x22, 0x11, 0x22)
    W["down_codes"][1] = 0x44  # expert 1's down weights are 2.0
    x = torch.ones(1, d, dtype=torch.bfloat16)
    idx, w = oracle_lib.route(np.array([[1.0, 0.0]], np.float32), 2)
    assert list(idx[0]) == [0, 1]
    out = oracle_lib.forward(_dims(d, 2, f, 2), W, _bits(x), idx, w, [0])
    y0 = 32 * (32.0 / (1.0 + math.exp(-32.0)) * 16.0)
    e = math.e
    assert np.allclose(out[0], y0 * (e / (e + 1) + 2 / (e + 1)), rtol=1e-14, atol=0)


def _torch_mxfp8(v: torch.Tensor) -> torch.Tensor:
    """MXFP8 round trip with torch's float8 cast as the element rounding."""
    blocks = v.reshape(-1, 32)
    amax = blocks.abs().amax(dim=1, keepdim=True)
    _, e = torch.frexp(amax)
    s = torch.where(amax > 0, (e - 1) - 8, torch.zeros_like(e)).clamp(-127, 127).to(torch.float64)
    q = (blocks / torch.exp2(s)).clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float64)
    return (q * torch.exp2(s)).reshape(v.shape)


_E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_by_search(v: float) -> int:
    """E2M1 code of v found by searching the eight magnitudes: the nearest one,
    ties to the even code, saturating at 6; the sign in bit 3."""
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(a - _E2M1_MAGNITUDES[c]), c % 2))
    return best | (8 if (v < 0 or (v == 0 and math.copysign(1.0, v) < 0)) else 0)


def _mxfp4_by_search(v: torch.Tensor) -> torch.Tensor:
    """MXFP4 round trip of an activation vector, the element rounding by search."""
    out = []
    for block in v.reshape(-1, 32).tolist():
        amax = max(abs(t) for t in block)
        s = 0 if amax == 0 else max(-127, min(127, (math.frexp(amax)[1] - 1) - 2))
        for t in block:
            c = _e2m1_by_search(math.ldexp(t, -s))
            out.append((-1.0 if c & 8 else 1.0) * _E2M1_MAGNITUDES[c & 7] * 2.0 ** s)
    return torch.tensor(out, dtype=torch.float64).reshape(v.shape)


def test_e2m1_encode_hand_values(oracle_lib):
    """Round to nearest, ties to the even code (OCP MX v1.0 conversion), worked by hand."""
    cases = [(0.0, 0), (0.25, 0), (0.26, 1), (0.5, 1), (0.75, 2), (1.0, 2), (1.25, 2), (1.3, 3), (1.75, 4),
             (2.5, 4), (2.6, 5), (3.5, 6), (5.0, 6), (5.5, 7), (6.0, 7), (100.0, 7), (-3.0, 0xD), (-0.2, 0x8)]
    for v, code in cases:
        assert oracle_lib.e2m1_encode(v) == code, v
    for c in range(16):  # every code value encodes to itself (-0 keeps its sign)
        val = (-1.0 if c & 8 else 1.0) * _E2M1_MAGNITUDES[c & 7]
        assert oracle_lib.e2m1_encode(val if c != 8 else -0.0) == c


def test_e2m1_encode_matches_search(oracle_lib):
    rng = np.random.default_rng(9)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), np.array([k / 4 for k in range(-28, 29)])])
    for v in vals:
        assert oracle_lib.e2m1_encode(float(v)) == _e2m1_by_search(float(v)), v


def test_mxfp4_activation_block_hand(oracle_lib):
    """amax 0.3: floor(log2 0.3) = -2, s = -4 (scale byte 123); 0.3 * 16 = 4.8 -> 4 (code 6), 0.1 * 16 = 1.6
    -> 1.5 (code 3), -0.02 * 16 = -0.32 -> -0.5 (code 9); an all-zero block has scale byte 127."""
    v = np.zeros(64)
    v[0], v[1], v[2] = 0.3, 0.1, -0.02
    codes, scales = oracle_lib.mxfp4_act(v)
    assert scales.tolist() == [123, 127]
    assert codes[:3].tolist() == [6, 3, 9] and not codes[3:].any()


@pytest.mark.parametrize("mode", ["exact", "mxfp8", "q2k", "mxfp4"])
def test_single_expert_matches_torch_float64(oracle_lib, mode):
    import oracle
    d, f = 256, 256
    wl = synth.Workload("pin", 3, d, 1, f, 1, 11, 11, "normal", "q2k" if mode == "q2k" else "mxfp4")
    W = _np_weights(synth.make_layer_weights(wl))
    x = synth.make_x(wl)
    dims = _dims(d, 1, f, 1)
    act = {"exact": oracle.ACT_EXACT, "mxfp8": oracle.ACT_MXFP8, "q2k": oracle.ACT_MXFP8_X_ONLY,
           "mxfp4": oracle.ACT_MXFP4}[mode]
    out = oracle_lib.forward(dims, W, _bits(x), np.zeros((3, 1), np.int32), np.ones((3, 1)), [0, 1, 2], act)
    wg, wu, wd = (torch.from_numpy(a) for a in oracle_lib.dequant_expert(dims, W, 0))
    xx = x.to(torch.float64)
    rt = _mxfp4_by_search if mode == "mxfp4" else _torch_mxfp8
    if mode != "exact":
        xx = torch.stack([rt(r) for r in xx])
    h = torch.nn.functional.silu(xx @ wg.T) * (xx @ wu.T)
    if mode in ("mxfp8", "mxfp4"):
        h = torch.stack([rt(r.to(torch.float32).to(torch.float64)) for r in h])
    ref = h @ wd.T
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-14 * float(ref.abs().max()))


@pytest.mark.parametrize("act", [0, 1, 2, 3])
def test_routed_equals_dense_mask(oracle_lib, act):
    wl = synth.WORKLOADS["tiny"]
    if act == 2:
        wl = synth.Workload("tinyq", 4, 256, 6, 256, 2, 0, 0, "perm", "q2k")
    W = _np_weights(synth.make_layer_weights(wl))
    inp = synth.make_inputs(wl)
    dims = _dims(wl.d, wl.E, wl.f, wl.k)
    idx, w = oracle_lib.route(inp["logits"].numpy(), wl.k)
    toks = list(range(wl.T))
    a = oracle_lib.forward(dims, W, _bits(inp["x"]), idx, w, toks, act)
    b = oracle_lib.forward_dense(dims, W, _bits(inp["x"]), idx, w, toks, act)
    scale = float(np.abs(b).max())
    assert scale > 0
    assert np.abs(a - b).max() <= 1e-13 * scale


def test_tiny_workload_has_no_ties_and_distinct_experts(oracle_lib):
    wl = synth.WORKLOADS["tiny"]
    lg = synth.make_logits(wl).numpy()
    for t in range(wl.T):
        assert len(set(lg[t].tolist())) == wl.E
    idx, w = oracle_lib.route(lg, wl.k)
    assert np.allclose(w.sum(1), 1.0, atol=1e-15)


# ----------------------------------------------------------------- fp16 and the Q2_K super-block stride
def test_half_golden(oracle_lib):
    g = GOLDEN["half"]
    for b, v in zip(g["bits"], g["values"]):
        got = oracle_lib.half(b)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(b), got, v)


def test_half_against_numpy_every_pattern(oracle_lib):
    # every finite binary16 pattern against numpy's float16 (a library routine)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(65536):
        r = float(ref[b])
        if math.isnan(r):
            assert math.isnan(oracle_lib.half(b))
        else:
            assert oracle_lib.half(b) == r, hex(b)


def _two_superblock_down(g, d):
    """Q2_K down weights [1][d][2][84] holding the hand-built rows of the pin
    (rows beyond them are all-zero blocks)."""
    dq = np.zeros((1, d, 2, 84), np.uint8)
    for r, row in enumerate(g["rows"]):
        for sb, blk in enumerate(row):
            dq[0, r, sb, 0:16] = blk["scale_bytes"]
            dq[0, r, sb, 16:80] = blk["qs_byte"]
            dq[0, r, sb, 80:82] = np.array([blk["d_bits"]], np.uint16).view(np.uint8)
            dq[0, r, sb, 82:84] = np.array([blk["dmin_bits"]], np.uint16).view(np.uint8)
    return dq


def test_q2k_two_superblocks_dequant(oracle_lib):
    """Weights at super-block index 1 of a 512-weight row (byte 84 of the row)
    and the row stride of 168 bytes, on hand-worked values."""
    g = GOLDEN["q2k_two_superblocks"]
    d, f = 32, 512
    W = _const_layer(d, f, 1, 0x22, 0x11, 0x22)
    del W["down_codes"], W["down_scales"]
    W["down_q2k"] = _two_superblock_down(g, d)
    _, _, wd = oracle_lib.dequant_expert(_dims(d, 1, f, 1), W, 0)
    for key, v in g["weights"].items():
        r, c = (int(s) for s in key.split(","))
        assert wd[r, c] == v, (key, wd[r, c], v)
    for r, s in enumerate(g["row_sums"]):
        assert wd[r].sum() == s
    assert not wd[len(g["rows"]):].any()


@pytest.mark.parametrize("mode", ["exact", "q2k_prefill"])
def test_q2k_two_superblocks_forward_closed_form(oracle_lib, mode):
    """The routed forward through the Q2_K row dot: gate = 1.0, up = 0.5 and
    x = 1 give g = 32, u = 16 and the same h for every feature, so
    y_m = h * (sum of row m's 512 weights), the hand-worked row sums."""
    import oracle
    g = GOLDEN["q2k_two_superblocks"]
    d, f = 32, 512
    W = _const_layer(d, f, 1, 0x22, 0x11, 0x22)
    del W["down_codes"], W["down_scales"]
    W["down_q2k"] = _two_superblock_down(g, d)
    x = torch.ones(1, d, dtype=torch.bfloat16)
    act = oracle.ACT_EXACT if mode == "exact" else oracle.ACT_MXFP8_X_ONLY
    out = oracle_lib.forward(_dims(d, 1, f, 1), W, _bits(x), np.zeros((1, 1), np.int32), np.ones((1, 1)), [0], act)
    h = 32.0 / (1.0 + math.exp(-32.0)) * 16.0
    want = np.zeros(d)
    want[:len(g["row_sums"])] = [h * s for s in g["row_sums"]]
    assert np.allclose(out[0], want, rtol=1e-14, atol=0)


# ----------------------------------------------------------------- router projection and shared expert
def _bf16_bits_np(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_router_logits_closed_form(oracle_lib):
    d = 64
    wr = np.zeros((3, d), np.float32)
    wr[0] = 1.0
    wr[1, ::2], wr[1, 1::2] = 1.0, -1.0
    wr[2, :32], wr[2, 32:] = 0.5, 2.0
    x = np.ones((2, d), np.float32)
    x[1, :32] = -1.0
    got = oracle_lib.router_logits(_bf16_bits_np(wr), _bf16_bits_np(x))
    # token 0: 64, 0, 16 + 64 = 80; token 1: -32 + 32 = 0, (-1 + 1)*16 + (1 - 1)*16 = 0, -16 + 64 = 48
    assert got.tolist() == [[64.0, 0.0, 80.0], [0.0, 0.0, 48.0]]


def test_router_logits_against_torch_float64(oracle_lib):
    g = torch.Generator().manual_seed(11)
    wr = (torch.randn(16, 256, generator=g) / 16).to(torch.bfloat16)
    x = torch.randn(5, 256, generator=g).to(torch.bfloat16)
    got = oracle_lib.router_logits(wr.view(torch.int16).numpy().view(np.uint16), x.view(torch.int16).numpy().view(np.uint16))
    ref = (x.double() @ wr.double().T).numpy()
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_shared_ffn_closed_form(oracle_lib):
    # gate 1.0, up 0.5, down 1.0, x = 1: g = 32, u = 16, h = bf16(fp32(silu(32) * 16)) = 512, y = 32 * 512
    d = fs = 32
    ones = np.ones((fs, d), np.float32)
    y = oracle_lib.shared_ffn(_bf16_bits_np(ones), _bf16_bits_np(0.5 * ones), _bf16_bits_np(ones),
                              _bf16_bits_np(np.ones((1, d), np.float32)), [0])
    assert y.tolist() == [[16384.0] * d]


def test_shared_ffn_against_torch_float64(oracle_lib):
    """The shared expert against torch: fp64 matmuls, SwiGLU, h rounded to fp32
    then bf16 by torch's casts (round to nearest even)."""
    g = torch.Generator().manual_seed(12)
    d, fs = 128, 96
    wg = (torch.randn(fs, d, generator=g) * 0.05).to(torch.bfloat16)
    wu = (torch.randn(fs, d, generator=g) * 0.05).to(torch.bfloat16)
    wd = (torch.randn(d, fs, generator=g) * 0.05).to(torch.bfloat16)
    x = torch.randn(3, d, generator=g).to(torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    y = oracle_lib.shared_ffn(bits(wg), bits(wu), bits(wd), bits(x), [0, 2])
    xs = x.double()[[0, 2]]
    gg, uu = xs @ wg.double().T, xs @ wu.double().T
    h = (torch.nn.functional.silu(gg) * uu).float().to(torch.bfloat16).double()
    ref = (h @ wd.double().T).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
