"""The round-up scale rule (MXG_SCALE_ROUND_UP) on the GPU quantizers,
bit-exact against the oracle's ``rule="round_up"``, and a GEMM fed operands
quantized that way.

Inputs put many block maxima on both sides of the rule's switch point (amax
mantissa above maxval's, 1.75 for E4M3 and 1.5 for E2M1), on exact powers of
two and in the subnormal range, where the OCP and round-up rules part."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

from gpu_util import bf16_to_dev, i32_to_dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


def _inputs(rng, shape):
    """Normal values, then each 32-block's first element replaced by a
    boundary maximum m * 2^k with m around 1.5 / 1.75 / 2 and k over a wide
    range (including subnormal BF16)."""
    x = synth.normal_bf16(rng, shape, std=1.0, outlier_frac=0.02)
    xf = synth.bf16_bits_to_f32(x)
    R, C = shape
    mant = rng.choice(np.array([1.0, 1.4921875, 1.5, 1.5078125, 1.7421875, 1.75, 1.7578125, 1.9921875],
                               dtype=np.float32), size=(R, C // 32))
    k = rng.integers(-135, 100, size=(R, C // 32)).astype(np.float32)
    sign = np.where(rng.random((R, C // 32)) < 0.5, -1.0, 1.0).astype(np.float32)
    head = sign * mant * np.float32(2.0) ** k
    xb = xf.reshape(R, C // 32, 32)
    xb = xb * (np.float32(2.0) ** np.minimum(k, 0)[..., None] * np.float32(0.5))   # keep the rest below the head
    xb[..., 0] = head
    return synth.f32_to_bf16_bits(xb.reshape(R, C))


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("shape", [(7, 96), (300, 512), (64, 4128)])
def test_rowwise_round_up(elem, shape):
    x = _inputs(np.random.default_rng(shape[0] + shape[1]), shape)
    op = _mxg().mx_quantize_rowwise(bf16_to_dev(x), elem, rule="round_up")
    torch.cuda.synchronize()
    d, s = oracle.quantize_mx_rowwise(x, elem, rule="round_up")
    assert np.array_equal(op.scale.cpu().numpy(), s)
    assert np.array_equal(op.data.cpu().numpy(), d)
    d0, s0 = oracle.quantize_mx_rowwise(x, elem)
    assert (s0 != s).any()          # the inputs do exercise the difference between the rules


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_packed_round_up(elem):
    splits = [0, 130, 1, 257]
    x = _inputs(np.random.default_rng(3), (sum(splits), 160))
    op = _mxg().mx_quantize_rowwise_packed(bf16_to_dev(x), elem, m_splits=i32_to_dev(splits), check=True,
                                           rule="round_up")
    d, s = oracle.quantize_mx_rowwise(x, elem, rule="round_up")
    assert np.array_equal(op.data.cpu().numpy(), d)
    ref = oracle.pack_scales_mma(s, splits)
    assert np.array_equal(op.scale.cpu().numpy()[: ref.size], ref)


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("dual", [False, True])
def test_colwise_and_dual_round_up(elem, dual):
    splits = np.array([37, 0, 5, 300, 64], dtype=np.int32)
    x = _inputs(np.random.default_rng(9), (int(splits.sum()), 256))
    mxg = _mxg()
    if dual:
        row, col, poff = mxg.mx_quantize_dual_segment_padded(bf16_to_dev(x), i32_to_dev(splits), 32, elem,
                                                             check=True, rule="round_up")
        rd, rs = oracle.quantize_mx_rowwise(x, elem, rule="round_up")
        assert np.array_equal(row.data.cpu().numpy(), rd)
        assert np.array_equal(row.scale.cpu().numpy(), rs)
    else:
        col, poff = mxg.mx_quantize_colwise_segment_padded(bf16_to_dev(x), i32_to_dev(splits), 32, elem,
                                                           check=True, rule="round_up")
    d, s, p = oracle.quantize_mx_colwise_segment_padded(x, splits, 32, elem, rule="round_up")
    spad = int(p[-1])
    cb = spad // 2 if elem == "e2m1" else spad
    assert np.array_equal(col.data.cpu().numpy()[:, :cb], d)
    assert np.array_equal(col.scale.cpu().numpy()[:, : spad // 32], s)


def test_fwd_on_round_up_operands():
    """A grouped forward on operands quantized with the round-up rule matches
    the oracle GEMM of the oracle's round-up operands (the GEMM itself does
    not depend on the rule)."""
    mxg = _mxg()
    splits = np.array([100, 0, 29, 300], dtype=np.int32)
    G, S, N, K = 4, int(splits.sum()), 96, 256
    rng = np.random.default_rng(5)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.02)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.02)
    A = mxg.mx_quantize_rowwise(bf16_to_dev(x), "e4m3", rule="round_up")
    W = mxg.mx_quantize_rowwise(bf16_to_dev(w), "e2m1", rule="round_up")
    Y = mxg.grouped_gemm_fwd(A, W, i32_to_dev(splits), N, check=True)
    ad, asc = oracle.quantize_mx_rowwise(x, "e4m3", rule="round_up")
    wd, wsc = oracle.quantize_mx_rowwise(w, "e2m1", rule="round_up")
    ref = oracle.grouped_fwd(oracle.dequantize_mx(ad, asc, "e4m3"),
                             oracle.dequantize_mx(oracle.unpack_e2m1(wd), wsc, "e2m1"), splits, N)
    oracle.assert_gemm_close(Y.float().cpu().numpy(), ref, "a8w4 fwd, round-up operands")
