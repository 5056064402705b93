"""Pins for the fp64 oracle against what the pages and the mathematics fix.

* I1  ReduceScatter + AllGather == AllReduce: the fused call on tp partials equals (a) one call on
      the exactly pre-summed tensor and (b) per-rank calls on each rank's reduced shard,
      concatenated (vllm-ascend SP/FlashComm notes §2.2, conclusion 1; §3.3 pad -> RS -> AG -> unpad).
* I2  per-token norm on shards == norm on the full tensor (same notes §2.2, conclusion 2).
* I3  per-token FP8 scales and NVFP4 block scales are shard-local; a per-tensor dynamic scale is
      not, which is why that mode is rejected (vLLM SP/AsyncTP/quant notes §四, correctness table).
* I4  padding rows come out as zero bytes whatever the padding inputs hold (PR #18671 §5.2, §5.3).
* I5  residual_out is the exact sum rounded once to bf16 (checked with rational arithmetic).
* I6  dequantised outputs are within half a code step of y (FP8 static / per-token, NVFP4).
* Closed forms of RMSNorm (constant row, one-hot row, the norm identity) and the library special
  case tp=1, no bias == torch.nn.functional.rms_norm in float64.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sequence_reduce_add_gb300 import synth

MODES = ["none", "fp8_static", "fp8_per_token", "nvfp4"]
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def ints(g, shape, lo, hi) -> torch.Tensor:
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


def rand_bf16(g, shape, std=1.0) -> torch.Tensor:
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def scale_for(mode):
    return {"fp8_static": 0.05, "nvfp4": 50.0}.get(mode)


def run(partials, residual, weight, bias, mode, T_valid, eps=1e-6, scale=None, **kw):
    if scale is None:
        scale = scale_for(mode)
    res = oracle.fused_reduce_norm(
        bits(partials), None if residual is None else bits(residual), bits(weight),
        None if bias is None else bits(bias), eps, mode, scale, T_valid, **kw)
    assert res["status"] == 0
    return res


def same(a: dict, b: dict):
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is None:
            assert b[k] is None
        else:
            assert np.array_equal(a[k], b[k]), k


def concat(parts: list[dict]) -> dict:
    return {k: (None if parts[0][k] is None else np.concatenate([p[k] for p in parts]))
            for k in ("out", "out_scales", "residual_out")}


# --------------------------------------------------------------------------- I1
@pytest.mark.parametrize("tp", [1, 2, 3, 4, 16])
@pytest.mark.parametrize("mode", MODES)
def test_rs_ag_equals_ar(tp, mode):
    g = torch.Generator().manual_seed(100 + tp)
    for S, H, pad in ((1, 16, 0), (3, 32, 2), (2, 16, 1)):
        T_pad = tp * S
        T_valid = max(T_pad - pad, 0)
        partials = ints(g, (tp, T_pad, H), -8, 8)
        residual = ints(g, (T_pad, H), -8, 8)
        bias = ints(g, (H,), -2, 2)
        weight = rand_bf16(g, (H,), 0.3) + 1
        fused = run(partials, residual, weight, bias, mode, T_valid)
        # AllReduce: the exact element-wise sum (small integers, exactly bf16), then the norm
        reduced = partials.double().sum(0).to(torch.bfloat16)
        assert torch.equal(reduced.double(), partials.double().sum(0))
        ar = run(reduced[None], residual, weight, bias, mode, T_valid)
        same(fused, ar)
        # ReduceScatter: rank r owns rows [r*S, (r+1)*S) of the sum; norm per shard; AllGather
        shards = []
        for r in range(tp):
            rows = slice(r * S, (r + 1) * S)
            valid = max(0, min(S, T_valid - r * S))
            shards.append(run(reduced[None, rows].contiguous(), residual[rows].contiguous(),
                              weight, bias, mode, valid))
        same(fused, concat(shards))


# --------------------------------------------------------------------------- I2
@pytest.mark.parametrize("mode", MODES)
def test_shard_norm_equals_full(mode):
    g = torch.Generator().manual_seed(7)
    tp, S, H = 4, 8, 64
    T_pad = tp * S
    T_valid = T_pad - 3
    partials = rand_bf16(g, (tp, T_pad, H), 0.5)
    residual = rand_bf16(g, (T_pad, H))
    weight, bias = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    full = run(partials, residual, weight, bias, mode, T_valid)
    shards = []
    for r in range(tp):
        rows = slice(r * S, (r + 1) * S)
        shards.append(run(partials[:, rows].contiguous(), residual[rows].contiguous(), weight,
                          bias, mode, max(0, min(S, T_valid - r * S))))
    same(full, concat(shards))


# --------------------------------------------------------------------------- library case
@pytest.mark.parametrize("H", [16, 256, 1000])
def test_tp1_no_bias_equals_torch_rms_norm(H):
    g = torch.Generator().manual_seed(H)
    T = 9
    x = rand_bf16(g, (1, T, H), 0.7)
    res = rand_bf16(g, (T, H))
    w = rand_bf16(g, (H,), 0.2) + 1
    eps = 1e-3
    got = run(x, res, w, None, "none", T, eps=eps, want_y=True)["y"]
    want = torch.nn.functional.rms_norm(x[0].double() + res.double(), (H,), w.double(),
                                        eps=float(np.float32(eps)))
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-13, atol=0)


# --------------------------------------------------------------------------- closed forms
def _rows_summing_to(g, target: torch.Tensor, tp: int):
    """Integer partials, residual and bias whose exact sum is ``target`` [T, H] (integers)."""
    T, H = target.shape
    partials = torch.randint(-6, 7, (tp, T, H), generator=g).double()
    residual = torch.randint(-6, 7, (T, H), generator=g).double()
    bias = torch.randint(-2, 3, (H,), generator=g).double()
    partials[0] = target - residual - bias - partials[1:].sum(0)
    assert partials.abs().max() <= 256  # exact in bf16
    return (partials.to(torch.bfloat16), residual.to(torch.bfloat16), bias.to(torch.bfloat16))


def test_constant_row_closed_form():
    g = torch.Generator().manual_seed(11)
    tp, H = 3, 48
    c = torch.tensor([5.0, -3.0, 0.0, 1.0, 17.0, -40.0])
    target = c[:, None].expand(-1, H).clone().double()
    partials, residual, bias = _rows_summing_to(g, target, tp)
    w = rand_bf16(g, (H,), 0.2) + 1
    eps = 0.25
    res = run(partials, residual, w, bias, "none", len(c), eps=eps, want_y=True)
    want = c.double()[:, None] / torch.sqrt(c.double()[:, None] ** 2 + eps) * w.double()[None]
    np.testing.assert_allclose(res["y"], want.numpy(), rtol=1e-14, atol=0)
    assert np.array_equal(res["out"], bits(want.to(torch.bfloat16)))
    assert np.array_equal(res["residual_out"], bits(target.to(torch.bfloat16)))


def test_one_hot_row_closed_form():
    g = torch.Generator().manual_seed(12)
    tp, H = 2, 64
    ks, cs = [0, 5, 63, 17], [3.0, -7.0, 1.0, 100.0]
    target = torch.zeros(len(ks), H).double()
    for i, (k, c) in enumerate(zip(ks, cs)):
        target[i, k] = c
    partials, residual, bias = _rows_summing_to(g, target, tp)
    w = rand_bf16(g, (H,), 0.2) + 1
    eps = 0.5
    y = run(partials, residual, w, bias, "none", len(ks), eps=eps, want_y=True)["y"]
    for i, (k, c) in enumerate(zip(ks, cs)):
        yk = np.sign(c) * np.sqrt(H) * float(w[k]) / np.sqrt(1 + H * eps / c ** 2)
        assert y[i, k] == pytest.approx(yk, rel=1e-14)
        assert np.all(np.delete(y[i], k) == 0)


def test_norm_identity_pins_eps_and_mean():
    # sum_j (y_j / w_j)^2 = H * ms / (ms + eps), ms = mean(h^2): exact rationals for integer h
    g = torch.Generator().manual_seed(13)
    tp, T, H = 4, 8, 40
    target = torch.randint(-9, 10, (T, H), generator=g).double()
    partials, residual, bias = _rows_summing_to(g, target, tp)
    w = rand_bf16(g, (H,), 0.2) + 1
    for eps in (1.0, 0.125, 8.0):
        y = run(partials, residual, w, bias, "none", T, eps=eps, want_y=True)["y"]
        lhs = ((y / w.double().numpy()[None]) ** 2).sum(1)
        for t in range(T):
            ms = Fraction(int((target[t] ** 2).sum().item()), H)
            assert lhs[t] == pytest.approx(float(H * ms / (ms + Fraction(eps))), rel=1e-13)


# --------------------------------------------------------------------------- I3
def test_per_token_and_block_scales_are_shard_local():
    g = torch.Generator().manual_seed(21)
    tp, S, H = 2, 4, 32
    T = tp * S
    partials = rand_bf16(g, (tp, T, H), 0.7)
    residual = rand_bf16(g, (T, H))
    residual[0, 3] = 60.0  # shard 0 holds the tensor-wide maximum
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    for mode in ("fp8_per_token", "nvfp4"):
        full = run(partials, residual, w, b, mode, T)
        per = [run(partials[:, r * S:(r + 1) * S].contiguous(),
                   residual[r * S:(r + 1) * S].contiguous(), w, b, mode, S) for r in range(tp)]
        assert np.array_equal(full["out_scales"], np.concatenate([p["out_scales"] for p in per]))
    # a per-tensor dynamic scale (max |y| over the tensor / 448) differs between shard 1 and
    # the whole tensor, so it cannot be computed on a shard: the oracle rejects that mode
    y = run(partials, residual, w, b, "none", T, want_y=True)["y"]
    assert np.abs(y[S:]).max() / 448 != np.abs(y).max() / 448
    st = oracle.check_args(1, tp, T, T, H, 2, 3, 4, 1e-6, "fp8_dynamic_per_tensor", None,
                           1 << 20, 1 << 21, 1 << 22)
    assert oracle.STATUS[st] == "unsupported"


# --------------------------------------------------------------------------- I4
@pytest.mark.parametrize("mode", MODES)
def test_padding_rows_are_zero_and_never_read(mode):
    g = torch.Generator().manual_seed(31)
    tp, T_pad, H, T_valid = 4, 12, 32, 9
    partials = rand_bf16(g, (tp, T_pad, H))
    residual = rand_bf16(g, (T_pad, H))
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    clean = run(partials, residual, w, b, mode, T_valid)
    partials[:, T_valid:] = float("nan")
    residual[T_valid:] = float("nan")
    dirty = run(partials, residual, w, b, mode, T_valid)
    same(clean, dirty)
    for k in ("out", "out_scales", "residual_out"):
        if dirty[k] is not None:
            assert not np.any(dirty[k][T_valid:].view(np.uint8))


def test_golden_shard_layout_padding():
    with open(os.path.join(GOLDEN, "shard_layout_tp16_t3500.json")) as f:
        gold = json.load(f)
    tp, T_pad, T, S = gold["tp"], gold["num_tokens_pad"], gold["num_tokens"], gold["local_tokens"]
    assert T_pad == S * tp and T_pad % tp == 0 and T_pad - T == len(gold["padding_rows"])
    g = torch.Generator().manual_seed(32)
    H = 16
    partials = ints(g, (tp, T_pad, H), -4, 4)
    residual = ints(g, (T_pad, H), -4, 4)
    residual[:, 0] = 100.0  # no valid row sums to zero
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    reduced = partials.double().sum(0).to(torch.bfloat16)  # exact: small integers
    partials[:, T:] = float("nan")
    residual[T:] = float("nan")
    full = run(partials, residual, w, b, "fp8_per_token", T)
    zero_rows = np.flatnonzero(~full["residual_out"].any(axis=1))
    assert list(zero_rows) == gold["padding_rows"]
    # each rank normalises its reduced 219-row shard after the ReduceScatter
    for r in range(tp):
        start = gold["shard_starts"][r]
        valid = gold["valid_tokens_per_shard"][r]
        assert valid == max(0, min(S, T - start))
        shard = run(reduced[None, start:start + S].contiguous(),
                    residual[start:start + S].contiguous(), w, b, "fp8_per_token", valid)
        assert np.array_equal(shard["out"], full["out"][start:start + S])
        assert np.array_equal(shard["out_scales"], full["out_scales"][start:start + S])
        assert np.count_nonzero(shard["residual_out"].any(axis=1)) == valid


# --------------------------------------------------------------------------- I5
def test_residual_out_is_exact_sum_rounded_once():
    g = torch.Generator().manual_seed(41)
    tp, T, H = 16, 16, 8
    partials = rand_bf16(g, (tp, T, H), 0.25)
    residual = rand_bf16(g, (T, H))
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    res = run(partials, residual, w, b, "none", T)
    got = res["residual_out"]
    for t in range(T):
        for j in range(H):
            exact = sum(Fraction(float(partials[r, t, j])) for r in range(tp))
            exact += Fraction(float(b[j])) + Fraction(float(residual[t, j]))
            code = int(got[t, j])
            v = Fraction(float(oracle.bf16_decode(np.array([code], np.uint16))[0]))
            for nb in (code - 1, code + 1):  # neighbours along the same sign's magnitude axis
                if (nb & 0x7FFF) == 0x7FFF or nb < 0 or nb > 0xFFFF or (nb ^ code) & 0x8000:
                    continue
                vn = Fraction(float(oracle.bf16_decode(np.array([nb], np.uint16))[0]))
                assert abs(v - exact) <= abs(vn - exact)
                if abs(v - exact) == abs(vn - exact):
                    assert code % 2 == 0


# --------------------------------------------------------------------------- I6
def _e4m3_half_step(v):
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -30))), -6)
    return 0.5 * 2.0 ** (e - 3)


def _e2m1_half_step(v):
    a = np.abs(v)
    return np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))


def _setup_quant(seed, T=6, H=64, tp=2):
    g = torch.Generator().manual_seed(seed)
    partials = rand_bf16(g, (tp, T, H), 0.7)
    residual = rand_bf16(g, (T, H))
    residual[:, 5] *= 50
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    return partials, residual, w, b, T


def test_fp8_static_dequant_within_half_step():
    partials, residual, w, b, T = _setup_quant(51)
    scale = 0.01  # the x50 channel saturates, the rest does not
    res = run(partials, residual, w, b, "fp8_static", T, scale=scale, want_y=True)
    v = res["y"] / np.float64(np.float32(scale))
    dq = oracle.e4m3_decode(res["out"].ravel()).reshape(v.shape)
    sat = np.abs(v) > 448
    assert np.all(dq[sat] == np.sign(v[sat]) * 448)
    assert np.all(np.abs(dq - v)[~sat] <= _e4m3_half_step(v[~sat]) * (1 + 1e-6))
    assert sat.any() and (~sat).any()


def test_fp8_per_token_scale_and_dequant():
    partials, residual, w, b, T = _setup_quant(52)
    res = run(partials, residual, w, b, "fp8_per_token", T, want_y=True)
    y, s = res["y"], res["out_scales"].astype(np.float64)
    amax = np.abs(y).max(1)
    np.testing.assert_allclose(s, amax / 448, rtol=2.0 ** -24)
    v = y / s[:, None]
    dq = oracle.e4m3_decode(res["out"].ravel()).reshape(v.shape)
    assert np.all(np.abs(dq - v) <= _e4m3_half_step(v) * (1 + 1e-6))
    assert np.all(np.abs(dq).max(1) == 448)  # each row's maximum lands on the top code


def test_nvfp4_block_scales_and_dequant():
    partials, residual, w, b, T = _setup_quant(53)
    gs = 60.0
    res = run(partials, residual, w, b, "nvfp4", T, scale=gs, want_y=True)
    y = res["y"]
    H = y.shape[1]
    sf = oracle.e4m3_decode(res["out_scales"].ravel()).reshape(T, H // 16)
    want_sf = gs * np.abs(y).reshape(T, H // 16, 16).max(2) / 6
    assert np.all(np.abs(sf - want_sf) <= _e4m3_half_step(want_sf) * (1 + 1e-6))
    packed = res["out"]
    codes = np.empty((T, H), np.uint8)
    codes[:, 0::2] = packed & 0xF  # element 2i: low nibble
    codes[:, 1::2] = packed >> 4
    q = oracle.e2m1_decode(codes.ravel()).reshape(T, H)
    v = y * gs / np.repeat(sf, 16, axis=1)
    sat = np.abs(v) > 6
    assert np.all(q[sat] == np.sign(v[sat]) * 6)
    assert np.all(np.abs(q - v)[~sat] <= _e2m1_half_step(v[~sat]) * (1 + 1e-6))


def test_zero_row_gives_zero_scale_and_codes():
    tp, T, H = 2, 2, 32
    partials = torch.zeros(tp, T, H, dtype=torch.bfloat16)
    residual = torch.zeros(T, H, dtype=torch.bfloat16)
    w = torch.ones(H, dtype=torch.bfloat16)
    for mode in ("fp8_per_token", "nvfp4", "fp8_static", "none"):
        res = run(partials, residual, w, None, mode, T)
        assert not res["out"].any()
        if res["out_scales"] is not None:
            assert not res["out_scales"].view(np.uint8).any()


# --------------------------------------------------------------------------- argument rules
def test_argument_rules():
    A = 1 << 20  # fake, never dereferenced, 16-byte aligned host addresses
    base = dict(partials_ptr=A, tp=4, T_pad=16, T_valid=13, H=64, residual_ptr=A * 8,
                weight_ptr=A * 9, bias_ptr=A * 10, eps=1e-6, mode="fp8_per_token", scale=None,
                out_ptr=A * 11, out_scales_ptr=A * 12, residual_out_ptr=A * 13)

    def st(**kw):
        return oracle.STATUS[oracle.check_args(**{**base, **kw})]

    assert st() == "ok"
    assert st(mode="fp8_dynamic_per_tensor") == "unsupported"
    assert st(mode=7) == "invalid_arg"
    assert st(tp=0) == "invalid_arg"
    assert st(T_pad=18) == "invalid_arg"          # not a multiple of tp
    assert st(T_valid=17) == "invalid_arg"
    assert st(T_valid=-1) == "invalid_arg"
    assert st(H=60) == "invalid_arg"
    assert st(H=72, mode="nvfp4", scale=1.0) == "invalid_arg"
    assert st(eps=0.0) == "invalid_arg"
    assert st(eps=float("inf")) == "invalid_arg"
    assert st(partials_ptr=None) == "invalid_arg"
    assert st(out_scales_ptr=None) == "invalid_arg"
    assert st(mode="fp8_static", scale=None, out_scales_ptr=None) == "invalid_arg"
    assert st(mode="fp8_static", scale=-1.0, out_scales_ptr=None) == "invalid_arg"
    assert st(residual_ptr=None) == "ok"          # the "First" pattern: no incoming residual
    assert st(bias_ptr=None) == "ok"
    assert st(residual_out_ptr=A * 8) == "ok"     # in place over the residual
    assert st(residual_out_ptr=A * 8 + 16) == "invalid_arg"  # partial overlap
    assert st(out_ptr=A + 64) == "invalid_arg"    # output inside the partials
    assert st(T_pad=0, T_valid=0, partials_ptr=None) == "ok"


# --------------------------------------------------------------------------- N3 extensions
def run_ex(partials, residual, weight, bias, mode, T_valid, partial_scale=1.0, addend=None,
           eps=1e-6, **kw):
    res = oracle.fused_reduce_norm(
        bits(partials), None if residual is None else bits(residual), bits(weight),
        None if bias is None else bits(bias), eps, mode, scale_for(mode), T_valid,
        partial_scale=partial_scale, addend=None if addend is None else bits(addend), **kw)
    assert res["status"] == 0
    return res


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("c", [0.5, 2.0, 0.25, -1.0])
def test_partial_scale_multiplies_each_partial_before_the_sum(mode, c):
    # a scale applied to every partial before the reduction (PR #18671 notes §5.3) is the
    # same as feeding already-scaled partials: exact here (integers times powers of two)
    g = torch.Generator().manual_seed(61)
    tp, T, H = 4, 8, 32
    partials = ints(g, (tp, T, H), -8, 8)
    residual, bias = ints(g, (T, H), -8, 8), ints(g, (H,), -2, 2)
    w = rand_bf16(g, (H,), 0.2) + 1
    scaled = (partials.double() * c).to(torch.bfloat16)
    assert torch.equal(scaled.double(), partials.double() * c)
    same(run_ex(partials, residual, w, bias, mode, T - 1, partial_scale=c),
         run_ex(scaled, residual, w, bias, mode, T - 1))


def test_partial_scale_matches_torch_rms_norm():
    g = torch.Generator().manual_seed(62)
    T, H, c = 9, 128, 1.0 / 3.0
    x = rand_bf16(g, (1, T, H), 0.7)
    res = rand_bf16(g, (T, H))
    w = rand_bf16(g, (H,), 0.2) + 1
    c32 = float(np.float32(c))
    y = run_ex(x, res, w, None, "none", T, partial_scale=c, eps=1e-3, want_y=True)["y"]
    want = torch.nn.functional.rms_norm(c32 * x[0].double() + res.double(), (H,), w.double(),
                                        eps=float(np.float32(1e-3)))
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-13, atol=0)


@pytest.mark.parametrize("mode", MODES)
def test_addend_is_added_like_the_residual(mode):
    g = torch.Generator().manual_seed(63)
    tp, T, H = 2, 6, 48
    partials = ints(g, (tp, T, H), -8, 8)
    residual, addend, bias = ints(g, (T, H), -8, 8), ints(g, (T, H), -8, 8), ints(g, (H,), -2, 2)
    w = rand_bf16(g, (H,), 0.2) + 1
    both = (residual.double() + addend.double()).to(torch.bfloat16)
    same(run_ex(partials, residual, w, bias, mode, T - 1, addend=addend),
         run_ex(partials, both, w, bias, mode, T - 1))
    # without a residual the addend alone plays its part
    same(run_ex(partials, None, w, bias, mode, T, addend=addend),
         run_ex(partials, addend, w, bias, mode, T))


@pytest.mark.parametrize("mode", MODES)
def test_addend_is_chunked_per_shard(mode):
    # reduce_scatter -> add(chunk(addend)[rank]) -> norm -> all_gather (SP/FlashComm notes §2.3)
    g = torch.Generator().manual_seed(64)
    tp, S, H = 4, 4, 32
    T = tp * S
    partials = rand_bf16(g, (tp, T, H), 0.5)
    residual, addend = rand_bf16(g, (T, H)), rand_bf16(g, (T, H), 0.3)
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    full = run_ex(partials, residual, w, b, mode, T - 3, partial_scale=0.75, addend=addend)
    shards = [run_ex(partials[:, r * S:(r + 1) * S].contiguous(),
                     residual[r * S:(r + 1) * S].contiguous(), w, b, mode,
                     max(0, min(S, T - 3 - r * S)), partial_scale=0.75,
                     addend=addend[r * S:(r + 1) * S].contiguous()) for r in range(tp)]
    same(full, concat(shards))


# --------------------------------------------------------------------------- N2 swizzled scales
@pytest.mark.parametrize("T,H", [(8, 64), (130, 80), (256, 1024), (3, 16)])
def test_swizzled_scales_hold_exactly_the_row_major_scales(T, H):
    """The 128x4-tile layout is a placement of the same block scales, padding zero: the swizzled
    buffer holds every row-major scale once plus (padded size - T*H/16) zero bytes, and the
    codes and y do not depend on the layout. (The placement map itself is checked on the GPU
    by cuBLASLt's block-scaled GEMM reading the library's output.)"""
    g = torch.Generator().manual_seed(T * 1000 + H)
    tp = 2
    T_pad = tp * -(-T // tp)
    partials = rand_bf16(g, (tp, T_pad, H), 0.7)
    residual = rand_bf16(g, (T_pad, H))
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    args = (bits(partials), bits(residual), bits(w), bits(b), 1e-6, "nvfp4", 60.0, T)
    flat = oracle.fused_reduce_norm(*args)
    swz = oracle.fused_reduce_norm(*args, scale_layout=1)
    assert flat["status"] == 0 and swz["status"] == 0
    assert np.array_equal(flat["out"], swz["out"])
    assert np.array_equal(flat["residual_out"], swz["residual_out"])
    rows, cols = -(-T_pad // 128) * 128, -(-(H // 16) // 4) * 4
    assert swz["out_scales"].shape == (rows * cols,)
    want = np.bincount(flat["out_scales"].ravel(), minlength=256)
    want[0] += rows * cols - T_pad * (H // 16)
    assert np.array_equal(np.bincount(swz["out_scales"], minlength=256), want)


def _torch_to_blocked():
    """PyTorch's own helper that rearranges a block-scale matrix into the 128x4-tile layout
    block-scaled GEMMs read (torch/testing/_internal/common_quantized.py, ``to_blocked``, written
    after the cuBLAS "1D block scaling factors layout" description). Its module imports test-only
    packages, so the two functions are taken from PyTorch's source file and run as they stand."""
    import ast
    path = os.path.join(os.path.dirname(torch.__file__), "testing", "_internal",
                        "common_quantized.py")
    if not os.path.exists(path):
        pytest.skip("this PyTorch has no common_quantized.py")
    with open(path) as f:
        tree = ast.parse(f.read())
    fns = [n for n in tree.body
           if isinstance(n, ast.FunctionDef) and n.name in ("ceil_div", "to_blocked")]
    if len(fns) != 2:
        pytest.skip("this PyTorch has no to_blocked helper")
    ns = {"torch": torch}
    exec(compile(ast.Module(body=fns, type_ignores=[]), path, "exec"), ns)
    return ns["to_blocked"]


@pytest.mark.parametrize("T,H", [(8, 64), (130, 80), (256, 1024), (3, 16), (300, 2000)])
def test_swizzled_scales_match_torch_blocked_layout(T, H):
    """The placement itself, pinned without a GPU: the oracle's swizzled scale buffer equals
    PyTorch's independent reshape/permute construction of the same layout applied to the oracle's
    row-major scales (padding bytes zero in both)."""
    to_blocked = _torch_to_blocked()
    g = torch.Generator().manual_seed(7 * T + H)
    tp = 2
    T_pad = tp * -(-T // tp)
    partials = rand_bf16(g, (tp, T_pad, H), 0.7)
    residual = rand_bf16(g, (T_pad, H))
    w, b = rand_bf16(g, (H,), 0.1) + 1, rand_bf16(g, (H,), 0.01)
    args = (bits(partials), bits(residual), bits(w), bits(b), 1e-6, "nvfp4", 60.0, T)
    flat = oracle.fused_reduce_norm(*args)
    swz = oracle.fused_reduce_norm(*args, scale_layout=1)
    assert flat["status"] == 0 and swz["status"] == 0
    want = to_blocked(torch.from_numpy(flat["out_scales"].reshape(T_pad, H // 16).copy()))
    assert np.array_equal(swz["out_scales"], want.numpy())
