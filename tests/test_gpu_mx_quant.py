"""Parity of the MXFP8 activation quantiser (moe_fp4_mxfp8_quantize, through
the C ABI) with the oracle's mxfp8_quantize.

Codes and scale bytes are integers, and both sides decide them exactly (the
inputs are bf16 values and the scales powers of two), so they must match bit
for bit: random bit patterns over the whole finite bf16 range (subnormals and
signed zeros included), exact E4M3 ties, saturating blocks, zero blocks, and
the activation shapes of the decode and prefill layers; blocks holding an
infinity or a NaN get the NaN scale byte and NaN codes.
"""
import numpy as np
import pytest

from oracle import moe_oracle as om
from oracle import mx_activations as mx
from moe_inputs import make_layer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that are exactly representable in bf16."""
    b = np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def bf16_exact(v: float) -> bool:
    b = np.array([v], dtype=np.float64).astype(np.float32)
    return b[0] == v and not (b.view(np.uint32)[0] & 0xFFFF)


def check(moe, bits: np.ndarray):
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = moe.mxfp8_quantize(x)
    torch.cuda.synchronize()
    ref_codes, ref_scales = mx.mxfp8_quantize(om.bf16_bits_to_f64(bits))
    got_s, got_c = scales.cpu().numpy(), codes.cpu().numpy()
    bad_s = np.nonzero(got_s != ref_scales)
    assert bad_s[0].size == 0, f"scale bytes differ at {bad_s[0][:4]}, {bad_s[1][:4]}"
    bad = np.nonzero(got_c != ref_codes)
    assert bad[0].size == 0, (f"codes differ at rows {bad[0][:4]} cols {bad[1][:4]}: got {got_c[bad][:4]}, "
                              f"want {ref_codes[bad][:4]}, x {om.bf16_bits_to_f64(bits)[bad][:4]}")


def random_finite_bits(rng, R, K):
    b = rng.integers(0, 1 << 16, size=(R, K), dtype=np.uint32)
    b = np.where(((b >> 7) & 0xFF) == 0xFF, b & 0x807F, b)     # inf / NaN exponent -> subnormal
    return b.astype(np.uint16)


@pytest.mark.parametrize("R,K", [(1, 32), (3, 64), (33, 4096), (7, 7168), (129, 2048)])
def test_random_bit_patterns(moe, R, K):
    rng = np.random.default_rng(R * 1000 + K)
    check(moe, random_finite_bits(rng, R, K))


def test_gaussian_rows_with_wide_row_scales(moe):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 1024)) * np.ldexp(1.0, rng.integers(-120, 120, size=(64, 1)))
    bits = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # truncation: any bf16 will do
    check(moe, bits)


def test_ties_saturation_zero_blocks_and_signed_zero(moe):
    table = mx.e4m3_decode(np.arange(128))              # non-negative codes
    fin = np.unique(table[np.isfinite(table)])
    mids = (fin[1:] + fin[:-1]) / 2.0                   # exact ties, 5 significant bits: bf16-exact
    rng = np.random.default_rng(6)
    rows = []
    for s in (-127, -60, 0, 37, 110):
        # ties that stay exact in bf16 at this scale (at 2^-127 the smallest ones fall off the subnormal grid)
        pool = mids[[bf16_exact(m * 2.0 ** s) for m in mids]]
        for trial in range(4):
            blk = rng.choice(pool, size=32) * rng.choice([-1.0, 1.0], size=32)
            blk[rng.integers(32)] = 448.0 if trial % 2 else 256.0     # block maximum in [256, 448]
            rows.append(blk * 2.0 ** s)
    sat = np.array([464.0, 472.0, 480.0, 496.0, 504.0, 510.0, -500.0, 300.0] * 4)   # (448, 512): saturate
    rows.append(sat * 2.0 ** -3)
    zero = np.zeros(32)
    zero[::3] = -0.0
    rows.append(zero)
    mixed = np.zeros(32)
    mixed[5] = -0.0
    mixed[9] = 1.0
    rows.append(mixed)
    bits = np.stack([f64_to_bf16_bits(r) for r in rows])
    check(moe, bits)


@pytest.mark.parametrize("T,d", [(32, 4096), (4608, 4096), (2048, 7168)])
def test_layer_activation_shapes(moe, T, d):
    """x of the decode, prefill and large layers (the same N(0, 1) bf16 recipe)"""
    L = make_layer(T=T, d=d, I=32, E=1, k=1, seed=T + d)
    check(moe, L.x_bf16)


def test_rows_zero_enqueues_nothing(moe):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    codes, scales = moe.mxfp8_quantize(x)
    assert codes.shape == (0, 64) and scales.shape == (0, 2)


def test_non_finite_blocks(moe):
    rng = np.random.default_rng(7)
    bits = random_finite_bits(rng, 4, 256)
    bits[0, 3] = 0x7F80    # +inf
    bits[1, 40] = 0xFF80   # -inf
    bits[2, 200] = 0x7FC1  # NaN
    bits[3, 31] = 0xFFFF   # NaN with the sign set
    bits[3, 32] = 0x7F80   # the next block too
    check(moe, bits)
