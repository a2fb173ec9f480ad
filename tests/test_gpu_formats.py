"""GPU: hardware format conversions and the device packers against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def test_cvt_decoders_exhaustive():
    a, b, _, _ = mk.probe_cvt()
    a = a.cpu().numpy().view(np.uint32)
    b = b.cpu().numpy().view(np.uint32)
    # every 16-bit pair of E4M3 codes: low byte -> low half
    lo, hi = _f16(a & 0xFFFF), _f16(a >> 16)
    for name, got, codes in (("lo", lo, np.arange(65536) & 0xFF), ("hi", hi, np.arange(65536) >> 8)):
        want = np.array([O.e4m3_value(c) for c in range(256)])[codes]
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), name
        assert np.array_equal(got[~nan], want[~nan]), name
    # every byte of two E2M1 codes: low nibble -> low half
    want_lo = np.array([O.e2m1_value(i & 0xF) for i in range(256)])
    want_hi = np.array([O.e2m1_value(i >> 4) for i in range(256)])
    assert np.array_equal(_f16(b & 0xFFFF), want_lo)
    assert np.array_equal(_f16(b >> 16), want_hi)


def test_cvt_encoders_match_oracle():
    rng = np.random.default_rng(0)
    e4_vals = sorted({O.e4m3_value(c) for c in range(0x7F)})
    e2_vals = sorted({O.e2m1_value(c) for c in range(8)})
    mids = [(x + y) / 2 for x, y in zip(e4_vals[:-1], e4_vals[1:])] + [(x + y) / 2 for x, y in zip(e2_vals[:-1], e2_vals[1:])]
    x = np.concatenate([rng.normal(0, 50, 20000), rng.uniform(-500, 500, 20000), rng.normal(0, 2, 20000),
                        np.array(mids), -np.array(mids), [0.0, -0.0, 1e-30, -1e-30, 448.0, 460.0, 6.0, 7.5]])
    if x.size % 2:
        x = np.append(x, 1.0)
    x = x.astype(np.float32)
    _, _, e4, e2 = mk.probe_cvt(torch.from_numpy(x).cuda())
    e4 = e4.cpu().numpy().view(np.uint16)
    e2 = e2.cpu().numpy()
    want4 = np.array([O.e4m3_encode(float(v)) for v in x], dtype=np.uint16)
    want2 = np.array([O.e2m1_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(e4 & 0xFF, want4[0::2]) and np.array_equal(e4 >> 8, want4[1::2])
    assert np.array_equal(e2 & 0xF, want2[0::2]) and np.array_equal(e2 >> 4, want2[1::2])


@pytest.mark.parametrize("shape", [(67, 320), (5, 1024), (1000, 3072)])
def test_pack_fp8_bit_exact(shape):
    w = S.random_matrix(*shape, seed=21)
    w[min(3, shape[0] - 1)] = 0
    codes, scales = mk.pack_fp8_row(mk.upload_bf16(w))
    oc, os_ = O.quant_fp8_row(w)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("shape", [(9, 96), (33, 1024), (1024, 3072)])
def test_pack_nvfp4_bit_exact(shape):
    w = S.random_matrix(*shape, seed=22)
    w[0, 16:32] = 0
    codes, bs, t = mk.pack_nvfp4(mk.upload_bf16(w))
    oc, ob, ot = O.quant_nvfp4(w)
    assert np.float32(t.item()).view(np.uint32) == np.float32(ot).view(np.uint32)
    assert np.array_equal(bs.cpu().numpy(), ob)
    assert np.array_equal(codes.cpu().numpy(), oc)



@pytest.mark.parametrize("shape", [(9, 96), (33, 1024), (3072, 1024)])
def test_pack_nvfp4_scale_search_bit_exact(shape):
    """The block-scale search packer against the oracle's, up to a full-size gate matrix."""
    w = S.random_matrix(*shape, seed=24)
    w[0, 16:32] = 0
    w[-1, -16:] = S.random_matrix(1, 16, seed=25, std=1e-5)[0]
    codes, bs, t = mk.pack_nvfp4(mk.upload_bf16(w), scale_search=True)
    oc, ob, ot = O.quant_nvfp4(w, scale_search=True)
    assert np.float32(t.item()).view(np.uint32) == np.float32(ot).view(np.uint32)
    assert np.array_equal(bs.cpu().numpy(), ob)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("shape", [(67, 320), (1000, 3072), (151936, 1024)])
def test_pack_fp8_bf16_scale_bit_exact(shape):
    """bf16 row scales against the oracle, up to the full tied embedding / LM head."""
    w = S.random_matrix(*shape, seed=26)
    w[min(3, shape[0] - 1)] = 0
    codes, scales = mk.pack_fp8_row(mk.upload_bf16(w), bf16_scale=True)
    oc, os_ = O.quant_fp8_row(w, bf16_scale=True)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oc)

def test_pack_full_size_lm_head_bit_exact():
    """The full 151,936 x 1024 tied matrix, FP8 per row, as the benchmark packs it."""
    w = S.random_matrix(151936, 1024, seed=23)
    codes, scales = mk.pack_fp8_row(mk.upload_bf16(w))
    oc, os_ = O.quant_fp8_row(w)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oc)
