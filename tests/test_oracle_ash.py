"""Pins of the oracle's adaptive rescaling (the per-channel powers of two of
the Adaptive Scale-Hadamard transform; TACO Core claim, Fig. 7).

* The rescaling is an exact multiply before the codec and after it: on
  inputs where x * down is exact (numpy, powers of two), the compress with
  the channel factors equals the plain compress of x * down (codes, scales,
  state), and the decompress equals the plain decompress times up.
* The reduce applies up after the inverse transform: equal to the plain
  reduce times up per channel; the fused TACO -> TACO reduce with equal
  blocks ignores the factors (the Hadamard-domain sums are already those of
  the rescaled tensors); with different blocks it is the reduce then the
  compress, both with the factors.
* The update rule on closed-form cases: equal channels keep factor 1; a
  channel 2^k above the others gets 2^-(k-2) for k >= 3; the factor is capped
  at 2^-3; empty channels keep 1; fewer than half outlying channels do not
  move the typical ones; the amax part is reset.
* The per-channel amax equals numpy's column max of |x|.
* On data with outlier channels the rescaled round trip loses less than the
  plain one (the purpose of the rescaling, TACO Fig. 8), and on data without
  outlier channels every factor is 1.
"""
import numpy as np
import pytest
import torch

import workloads


def _chan(orc, cols, exps):
    c = orc.new_chan_state(cols)
    e = np.asarray(exps, dtype=np.float64)
    c[:cols] = np.exp2(-e).astype(np.float32)
    c[cols:2 * cols] = np.exp2(e).astype(np.float32)
    return c


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("mode", [0, 1])
def test_rescaled_compress_is_the_plain_compress_of_x_times_down(orc, B, mode):
    rng = np.random.default_rng(B + mode)
    rows, cols = 6, 512
    x = (rng.standard_normal((rows, cols)) * 0.03).astype(np.float32)
    exps = rng.integers(0, 6, size=cols)
    x[:, exps > 3] *= 40
    chan = _chan(orc, cols, exps)
    xd = (x.astype(np.float64) * np.exp2(-exps.astype(np.float64))[None, :]).astype(np.float32)
    assert np.array_equal(xd.astype(np.float64), x.astype(np.float64) * np.exp2(-exps)[None, :])   # exact
    st1 = np.array([0.01, 0.0], np.float32)
    st2 = st1.copy()
    a = orc.compress(orc.TACO_FP8, B, x.reshape(-1), orc.FP32, 1, rows, cols, st1, mode, chan=chan)
    b = orc.compress(orc.TACO_FP8, B, xd.reshape(-1), orc.FP32, 1, rows, cols, st2, mode)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(st1, st2)
    ya = orc.decompress(orc.TACO_FP8, B, a[0], a[1], None, st1, 1, rows, cols, orc.FP32, chan=chan)
    yb = orc.decompress(orc.TACO_FP8, B, b[0], b[1], None, st2, 1, rows, cols, orc.FP32).reshape(rows, cols)
    want = (yb.astype(np.float64) * np.exp2(exps)[None, :]).astype(np.float32)
    assert np.array_equal(ya.reshape(rows, cols).view(np.uint32), want.view(np.uint32))


def test_rescaled_reduce_and_fused_reduce(orc):
    rng = np.random.default_rng(3)
    n, rows, cols, B = 3, 8, 512, 128
    exps = rng.integers(0, 5, size=cols)
    chan = _chan(orc, cols, exps)
    shards = []
    for r in range(n):
        x = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
        x[:, exps > 2] *= 30
        st = np.zeros(2, np.float32)
        c, s, _ = orc.compress(orc.TACO_FP8, B, x.reshape(-1), orc.FP32, 1, rows, cols, st, orc.CURRENT, chan=chan)
        shards.append((c, s, None, st))
    plain = orc.reduce(orc.TACO_FP8, B, shards, rows, cols).reshape(rows, cols)
    resc = orc.reduce(orc.TACO_FP8, B, shards, rows, cols, chan=chan).reshape(rows, cols)
    want = (plain.astype(np.float64) * np.exp2(exps)[None, :]).astype(np.float32)
    assert np.array_equal(resc.view(np.uint32), want.view(np.uint32))
    # equal blocks: the Hadamard-domain path, the factors do not enter
    s1 = np.array([0.02, 0.0, 0.03, 0.0], np.float32)
    s2 = s1.copy()
    f1 = orc.reduce_requant(orc.TACO_FP8, B, shards, rows, cols, 0, rows, orc.TACO_FP8, B, 2, s1, orc.DELAYED,
                            chan=chan)
    f2 = orc.reduce_requant(orc.TACO_FP8, B, shards, rows, cols, 0, rows, orc.TACO_FP8, B, 2, s2, orc.DELAYED)
    assert all(np.array_equal(a, b) for a, b in zip(f1[:2], f2[:2])) and np.array_equal(s1, s2)
    # other blocks: reduce (times up) then compress (times down)
    s3 = np.array([0.02, 0.0, 0.03, 0.0], np.float32)
    s4 = s3.copy()
    g1 = orc.reduce_requant(orc.TACO_FP8, B, shards, rows, cols, 0, rows, orc.TACO_FP8, 256, 2, s3, orc.DELAYED,
                            chan=chan)
    g2 = orc.compress(orc.TACO_FP8, 256, resc.reshape(-1), orc.FP32, 2, rows // 2, cols, s4, orc.DELAYED, chan=chan)
    assert all(np.array_equal(a, b) for a, b in zip(g1[:2], g2[:2])) and np.array_equal(s3, s4)
    # the factors only go with TACO
    with pytest.raises(ValueError):
        orc.compress(orc.INT8_SYM, 64, np.zeros(cols, np.float32), orc.FP32, 1, 1, cols, chan=chan)


def _update(orc, amax):
    cols = len(amax)
    c = orc.new_chan_state(cols)
    c[2 * cols:] = np.asarray(amax, np.float32)
    orc.ash_update(c, cols)
    down, up, am = c[:cols], c[cols:2 * cols], c[2 * cols:]
    assert np.all(am == 0)
    assert np.array_equal(down.astype(np.float64) * up.astype(np.float64), np.ones(cols))
    e = np.log2(up.astype(np.float64))
    assert np.array_equal(e, np.round(e))                    # powers of two
    return e.astype(int)


def test_update_rule_closed_forms(orc):
    # equal channels: no rescaling
    assert np.all(_update(orc, [0.3] * 16) == 0)
    # one channel 2^k above the others (same mantissa): 2^-min(3, k-2) for k >= 3
    for k in range(0, 12):
        e = _update(orc, [0.75] * 15 + [0.75 * 2.0 ** k])
        assert np.all(e[:15] == 0) and e[15] == min(3, max(0, k - 2)), k
    # the cap
    assert _update(orc, [1.0] * 9 + [2.0 ** 40])[9] == 3
    # empty channels keep factor 1 and do not count for the median
    e = _update(orc, [0.0] * 10 + [1.0, 1.0, 1.0, 16.0])
    assert list(e) == [0] * 13 + [2]
    # fewer than half outlying channels leave the typical ones alone
    am = np.full(64, 0.01)
    am[:31] = 0.3                       # exponent -2 against -7: 5 above
    e = _update(orc, am)
    assert np.all(e[31:] == 0) and np.all(e[:31] == 3)
    am[:31] = 0.07                      # exponent -4: 3 above
    e = _update(orc, am)
    assert np.all(e[31:] == 0) and np.all(e[:31] == 1)


def test_channel_amax_is_the_column_max(orc):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((3, 7, 256)) * np.exp(rng.uniform(-3, 3, (1, 1, 256)))).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    c = orc.new_chan_state(256)
    c[512:] = 0.5                                            # max-accumulated onto the old values
    orc.channel_amax(bits, orc.BF16, 3, 7, 256, c)
    ref = np.maximum(np.abs(xb.float().numpy()).reshape(-1, 256).max(axis=0), 0.5).astype(np.float32)
    assert np.array_equal(c[512:], ref)
    assert np.all(c[:512] == 1.0)


@pytest.mark.parametrize("name,better", [("gpt_tp", True), ("flash_int4", True), ("equarx_int8", False),
                                         ("qwen_grad", False)])
def test_rescaling_helps_outlier_channels(orc, name, better):
    w = workloads.WORKLOADS[name]
    x = workloads.make_rank_inputs(w, rows=256, ranks=1)[0]
    bits = x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    dt = orc.BF16 if w.dtype == "bf16" else orc.FP16
    R, C = 256, w.cols
    chan = orc.new_chan_state(C)
    orc.channel_amax(bits, dt, 1, R, C, chan)
    orc.ash_update(chan, C)
    xf = x.float().numpy().astype(np.float64)

    def mse(ch):
        st = np.zeros(2, np.float32)
        c, s, _ = orc.compress(orc.TACO_FP8, 128, bits, dt, 1, R, C, st, orc.CURRENT, chan=ch)
        y = orc.decompress(orc.TACO_FP8, 128, c, s, None, st, 1, R, C, orc.FP32, chan=ch).reshape(R, C)
        return float(((y - xf) ** 2).mean())

    if better:
        assert np.any(chan[:C] < 1.0)
        assert mse(chan) < 0.8 * mse(None)
    else:
        assert np.all(chan[:C] == 1.0)
        assert mse(chan) == mse(None)
