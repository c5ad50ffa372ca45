"""FP8 (E4M3) block quantisation and the FP8 forward through the C ABI, against the oracle."""

import numpy as np
import pytest

import oracle
from oracle import fp8 as F8
from helpers import (TOL_FP8_ACC_U, TOL_FP8_O_MAXABS_OF_VMAX, TOL_FP8_O_RELRMS, TOL_L_MAXABS, max_abs,
                     rel_rms, to_device, to_f64)
from exact_tiled_attention_07_gb300.inputs import round_to_dtype, to_float64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _draw(shape, seed, spread=True):
    """N(0,1) values, each 128-row block of a head scaled by its own factor in [1e-3, 1e2]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(shape, dtype=np.float32)
    if spread:
        nb = (shape[-2] + 127) // 128
        f = np.exp(rng.uniform(np.log(1e-3), np.log(1e2), size=shape[:-2] + (nb,))).astype(np.float32)
        x *= np.repeat(f, 128, axis=-1)[..., : shape[-2], None]
    return x


def _codes_to_bytes(codes):
    """Oracle code values (exact E4M3 values) -> their bytes, by torch's float8 conversion."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("n", [1, 127, 128, 300])
def test_quantize_codes_and_scales_are_bit_exact(fa, dtype, d, n):
    x = round_to_dtype(_draw((2, 3, n, d), 10 + d + n), dtype)
    x64 = to_float64(x, dtype)
    codes, scales = F8.quantize_blocks(x64)
    x8, sc = fa.quantize_fp8(to_device(x, dtype))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sc.cpu().numpy(), scales)
    np.testing.assert_array_equal(x8.cpu().numpy(), _codes_to_bytes(codes).numpy())


def test_quantize_all_zero_block_and_saturation(fa):
    x = np.zeros((1, 1, 256, 128), dtype=np.float32)
    x[0, 0, 128:, :] = np.linspace(-3.0, 5.0, 128 * 128, dtype=np.float32).reshape(128, 128)
    x8, sc = fa.quantize_fp8(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert sc[0, 0, 0].item() == 1.0 and not x8[0, 0, :128].any()
    codes, scales = F8.quantize_blocks(x)
    assert sc[0, 0, 1].item() == scales[0, 0, 1]
    np.testing.assert_array_equal(x8.cpu().numpy(), _codes_to_bytes(codes).numpy())
    # the block maximum maps to 448 = byte 0x7E
    assert int(x8[0, 0, 255, 127].item()) == 0x7E


def test_quantize_quotients_at_and_beside_e4m3_midpoints(fa):
    """Quotients x / s on, and up to 6 fp32 ulps either side of, every midpoint between two
    E4M3 values (where the rounding decision flips, including the subnormal range), with a scale
    that is not a power of two: the codes must still be those of the correctly rounded fp32
    quotient, bit for bit."""
    amax = np.float32(300.7)
    s = np.float32(amax / np.float32(F8.E4M3_MAX))  # the scale this block's maximum gives
    vals = F8.e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2
    xs = []
    for m in mids:
        x0 = np.float32(np.float64(m) * np.float64(s))
        lo = hi = x0
        xs.append(x0)
        for _ in range(6):
            lo = np.nextafter(lo, np.float32(-np.inf), dtype=np.float32)
            hi = np.nextafter(hi, np.float32(np.inf), dtype=np.float32)
            xs.extend([lo, hi])
    xs = np.array(xs, dtype=np.float32)
    assert np.abs(xs).max() < amax
    block = np.zeros(128 * 128, dtype=np.float32)
    block[0] = amax
    block[1:1 + xs.size] = xs
    block[1 + xs.size:1 + 2 * xs.size] = -xs
    x = block.reshape(1, 1, 128, 128)
    codes, scales = F8.quantize_blocks(x)
    assert scales[0, 0, 0] == s
    x8, sc = fa.quantize_fp8(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert sc[0, 0, 0].item() == s
    np.testing.assert_array_equal(x8.cpu().numpy(), _codes_to_bytes(codes).numpy())


def _fp8_case(b, h, n, seed, spread=True, d=128):
    q, k, v = (_draw((b, h, n, d), seed + i, spread) for i in range(3))
    qc, qs = F8.quantize_blocks(q)
    kc, ks = F8.quantize_blocks(k)
    vc, vs = F8.quantize_blocks(v)
    dev = [_codes_to_bytes(c).cuda() for c in (qc, kc, vc)] + [torch.from_numpy(s).cuda() for s in (qs, ks, vs)]
    return (qc, qs, kc, ks, vc, vs), dev


def _abs_dot_rows(q, k, scale, causal, rows):
    """max_j tau sum_k |q_ik| |k_jk| over the visible keys j of each row (b, h, i): the size of
    the largest sum of products the tensor core forms for that row."""
    out = []
    for b, h, i in rows:
        a = scale * (np.abs(k[b, h]) @ np.abs(q[b, h, i]))
        out.append((a[: i + 1] if causal else a).max())
    return np.array(out)


def _check_l(gl, l_ref, absdot):
    err = np.abs(np.asarray(gl, np.float64) - l_ref)
    bound = TOL_L_MAXABS + TOL_FP8_ACC_U * absdot
    assert np.all(err <= bound), (err.max(), float(((err - TOL_L_MAXABS) / absdot).max()))


def _check_o(go, o_ref, vmax):
    assert rel_rms(go, o_ref) <= TOL_FP8_O_RELRMS, rel_rms(go, o_ref)
    assert max_abs(go, o_ref) <= TOL_FP8_O_MAXABS_OF_VMAX * vmax + 1e-3


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [128, 129, 300, 1000])
@pytest.mark.parametrize("out", ["bf16", "fp16"])
def test_fp8_forward_matches_attention_on_dequantised_inputs(fa, d, causal, n, out):
    host, dev = _fp8_case(2, 2, n, 50 + n + causal + d, d=d)
    scale = d ** -0.5
    odt = torch.bfloat16 if out == "bf16" else torch.float16
    o, lse = fa.attention_forward_fp8(*dev[:3], *dev[3:], scale=scale, causal=causal, out_dtype=odt)
    fa.fa_check_device_error()
    o_ref, l_ref = F8.attn_fwd64_fp8(*host, scale, causal)
    vmax = np.abs(F8.dequantize_blocks(host[4], host[5])).max()
    _check_o(to_f64(o), o_ref, vmax)
    rows = list(np.ndindex(2, 2, n))
    deq = [F8.dequantize_blocks(host[2 * i], host[2 * i + 1]) for i in range(2)]
    _check_l(to_f64(lse).reshape(-1), l_ref.reshape(-1), _abs_dot_rows(deq[0], deq[1], scale, causal, rows))


def _exact_values(shape, seed):
    """code x 2^-8 with codes in +-{256, 288, ..., 448} (the E4M3 values of exponent 8: 1.0 to
    1.75 x 2^8) and a +448 in every 128-row block, so every block scale is exactly 2^-8, every
    value quantises to its own code and every product of two codes is a multiple of 1024.  The
    first row of each block is positive with codes of at least 384, so a group of 32 products
    of two such rows sums to between 4608 and 6272 times 1024: 13 significant bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = (rng.integers(8, 15, size=shape) * 32 * rng.choice([-1, 1], size=shape)).astype(np.float32)
    codes[..., ::128, :] = rng.integers(12, 15, size=codes[..., ::128, :].shape) * 32
    codes[..., ::128, 0] = 448.0
    return codes * np.float32(2.0 ** -8)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_exact_sums_meet_the_plain_l_tolerance(fa, causal, d):
    """Inputs whose products and sums are exact in 13 significant bits: S has no rounding beyond
    the tensor core's accumulation, so L must meet the plain 1e-3 (no score-size term); O keeps
    the tolerance of the E4M3 rounding of P."""
    b, h, n = 2, 2, 300
    q, k, v = (_exact_values((b, h, n, d), 500 + i + d) for i in range(3))
    host, dev = [], []
    for t in (q, k, v):
        c, sc = F8.quantize_blocks(t)
        assert (sc == 2.0 ** -8).all() and np.array_equal(c * 2.0 ** -8, t)
        host += [c, sc]
    x8 = [fa.quantize_fp8(torch.from_numpy(t).cuda()) for t in (q, k, v)]
    torch.cuda.synchronize()
    for (c8, s8), c, sc in zip(x8, host[0::2], host[1::2]):
        np.testing.assert_array_equal(c8.cpu().numpy(), _codes_to_bytes(c).numpy())
        np.testing.assert_array_equal(s8.cpu().numpy(), sc)
    scale = d ** -0.5
    o, lse = fa.attention_forward_fp8(*(c8 for c8, _ in x8), *(s8 for _, s8 in x8), scale=scale, causal=causal)
    fa.fa_check_device_error()
    o_ref, l_ref = F8.attn_fwd64_fp8(*host, scale, causal)
    assert max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS, max_abs(to_f64(lse), l_ref)
    _check_o(to_f64(o), o_ref, np.abs(v).max())


def test_fp8_forward_unit_scales_and_causal_tiles(fa):
    # uniform magnitudes: every block scale close to the others; causal tile count T (T + 1) / 2
    host, dev = _fp8_case(1, 3, 1000, 90, spread=False)
    fa.fa_tile_counter(reset=True)
    o, lse = fa.attention_forward_fp8(*dev[:3], *dev[3:], causal=True)
    torch.cuda.synchronize()
    t = (1000 + 127) // 128
    assert fa.fa_tile_counter() == 3 * t * (t + 1) // 2
    o_ref, l_ref = F8.attn_fwd64_fp8(*host, 128 ** -0.5, True)
    _check_o(to_f64(o), o_ref, np.abs(F8.dequantize_blocks(host[4], host[5])).max())
    assert max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS


def test_fp8_forward_full_size_sampled_rows(fa):
    # the causal LM shape (B 8, H 16, N 4096, d 128), sampled rows against the oracle
    b, h, n = 8, 16, 4096
    host, dev = _fp8_case(b, h, n, 123, spread=False)
    o, lse = fa.attention_forward_fp8(*dev[:3], *dev[3:], causal=True)
    fa.fa_check_device_error()
    rng = np.random.default_rng(5)
    samples = np.stack([rng.integers(0, b, 48), rng.integers(0, h, 48), rng.integers(0, n, 48)], axis=1)
    samples = np.concatenate([samples, [[0, 0, 0], [7, 15, n - 1], [3, 4, 128], [5, 9, 127]]])
    deq = [F8.dequantize_blocks(host[2 * i], host[2 * i + 1]) for i in range(3)]
    o_ref, l_ref = oracle.attn_fwd64_rows(*deq, 128 ** -0.5, True, samples)
    go, gl = to_f64(o), to_f64(lse)
    got_o = np.stack([go[bb, hh, ii] for bb, hh, ii in samples])
    got_l = np.array([gl[bb, hh, ii] for bb, hh, ii in samples])
    _check_o(got_o, o_ref, np.abs(deq[2]).max())
    _check_l(got_l, l_ref, _abs_dot_rows(deq[0], deq[1], 128 ** -0.5, True, samples))


def test_fp8_argument_checks(fa):
    for d in (32, 96):
        z = torch.zeros((1, 1, 128, d), dtype=torch.uint8, device="cuda")
        s = torch.ones(1, dtype=torch.float32, device="cuda")
        with pytest.raises(fa.FAError, match="d in"):
            fa.attention_forward_fp8(z, z, z, s, s, s)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h,hkv", [(4, 2), (4, 1)])
def test_fp8_forward_grouped_query_heads(fa, causal, h, hkv, d):
    """fa_fwd_fp8_gqa: query head i reads key/value head i / (H / Hkv); against the fp64 oracle
    of grouped-query attention on the dequantised inputs."""
    n = 300
    q = _draw((2, h, n, d), 70 + h + hkv + d)
    k, v = (_draw((2, hkv, n, d), 80 + i + hkv + d) for i in range(2))
    (qc, qs), (kc, ks), (vc, vs) = (F8.quantize_blocks(t) for t in (q, k, v))
    dev = [_codes_to_bytes(c).cuda() for c in (qc, kc, vc)] + [torch.from_numpy(x).cuda() for x in (qs, ks, vs)]
    scale = d ** -0.5
    o, lse = fa.attention_forward_fp8(*dev[:3], *dev[3:], scale=scale, causal=causal)
    fa.fa_check_device_error()
    deq = [F8.dequantize_blocks(c, x) for c, x in ((qc, qs), (kc, ks), (vc, vs))]
    from oracle import gqa as G
    o_ref, l_ref = G.attn_fwd64_gqa(deq[0], deq[1], deq[2], scale, causal)
    _check_o(to_f64(o), o_ref, np.abs(deq[2]).max())
    kx = np.repeat(deq[1], h // hkv, axis=1)
    rows = list(np.ndindex(2, h, n))
    _check_l(to_f64(lse).reshape(-1), l_ref.reshape(-1), _abs_dot_rows(deq[0], kx, scale, causal, rows))


def test_fp8_forward_d64_gpt2_medium_shape_sampled_rows(fa):
    # the GPT-2-medium attention shape (B 64, H 16, N 1024, d 64), sampled rows against the oracle
    b, h, n, d = 64, 16, 1024, 64
    host, dev = _fp8_case(b, h, n, 321, spread=False, d=d)
    o, lse = fa.attention_forward_fp8(*dev[:3], *dev[3:], causal=False)
    fa.fa_check_device_error()
    rng = np.random.default_rng(6)
    samples = np.stack([rng.integers(0, b, 48), rng.integers(0, h, 48), rng.integers(0, n, 48)], axis=1)
    samples = np.concatenate([samples, [[0, 0, 0], [b - 1, h - 1, n - 1], [3, 4, 128], [5, 9, 127]]])
    deq = [F8.dequantize_blocks(host[2 * i], host[2 * i + 1]) for i in range(3)]
    o_ref, l_ref = oracle.attn_fwd64_rows(*deq, d ** -0.5, False, samples)
    go, gl = to_f64(o), to_f64(lse)
    got_o = np.stack([go[bb, hh, ii] for bb, hh, ii in samples])
    got_l = np.array([gl[bb, hh, ii] for bb, hh, ii in samples])
    _check_o(got_o, o_ref, np.abs(deq[2]).max())
    _check_l(got_l, l_ref, _abs_dot_rows(deq[0], deq[1], d ** -0.5, False, samples))


def test_fp8_forward_d256_head_dim_256_shape_sampled_rows(fa):
    """The large-head-dimension shape (B 4, H 16, N 16384, d 256, non-causal), sampled rows.  The
    device quantises the whole problem (its codes are checked bit for bit against the oracle's
    quantiser above); the oracle quantises, from the same fp32 values, only the heads it samples."""
    b, h, n, d = 4, 16, 16384, 256
    x = [_draw((b, h, n, d), 654 + i, spread=False) for i in range(3)]
    x8 = [fa.quantize_fp8(torch.from_numpy(t).cuda()) for t in x]
    o, lse = fa.attention_forward_fp8(*(c for c, _ in x8), *(s for _, s in x8), causal=False)
    fa.fa_check_device_error()
    del x8
    rng = np.random.default_rng(7)
    samples = np.stack([rng.integers(0, b, 40), rng.integers(0, h, 40), rng.integers(0, n, 40)], axis=1)
    samples = np.concatenate([samples, [[0, 0, 0], [b - 1, h - 1, n - 1], [2, 3, 128], [1, 7, 127]]])
    go, gl = to_f64(o), to_f64(lse)
    got_o = np.stack([go[bb, hh, ii] for bb, hh, ii in samples])
    got_l = np.array([gl[bb, hh, ii] for bb, hh, ii in samples])
    o_ref, l_ref = np.zeros_like(got_o), np.zeros_like(got_l)
    absdot, vmax = np.zeros_like(got_l), 0.0
    for bb, hh in sorted({(int(p), int(q)) for p, q, _ in samples}):
        idx = np.nonzero((samples[:, 0] == bb) & (samples[:, 1] == hh))[0]
        rows = np.stack([np.zeros_like(idx), np.zeros_like(idx), samples[idx, 2]], axis=1)
        deq = [F8.dequantize_blocks(*F8.quantize_blocks(t[bb, hh][None, None])) for t in x]
        o_ref[idx], l_ref[idx] = oracle.attn_fwd64_rows(*deq, d ** -0.5, False, rows)
        absdot[idx] = _abs_dot_rows(deq[0], deq[1], d ** -0.5, False, rows)
        vmax = max(vmax, float(np.abs(deq[2]).max()))
    _check_o(got_o, o_ref, vmax)
    _check_l(got_l, l_ref, absdot)
