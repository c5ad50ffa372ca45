"""Block-sparse and sliding-window masks through the C ABI vs the fp64 oracle."""

import numpy as np
import pytest

from oracle import gqa as G
from oracle import masks as MK
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import TOL_GRAD_RELRMS, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, max_abs, rel_rms, to_device, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _block_mask(heads, n, density, seed, empty_row=None):
    nb = (n + 127) // 128
    rng = np.random.default_rng(seed)
    bm = (rng.random((heads, nb, nb)) < density).astype(np.uint8)
    if empty_row is not None:
        bm[:, empty_row, :] = 0  # those query rows see no key
    return bm


def _check(fa, w, window=0, bm=None, backward=True):
    """Forward (and backward) of workload w with the mask, element-wise against the oracle."""
    x = make_inputs(w, with_do=backward)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    bm_dev = None if bm is None else torch.from_numpy(np.ascontiguousarray(bm[0] if bm.shape[0] == 1 else bm)).cuda()
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale, window=window,
                                  block_mask=bm_dev)
    if backward:
        dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=w.causal,
                                           scale=w.scale, window=window, block_mask=bm_dev)
    fa.fa_check_device_error()
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    ke, ve = G.expand_kv(x64["k"], w.H), G.expand_kv(x64["v"], w.H)
    vis = MK.visible_mask(w.N, w.causal, window, bm)
    o_ref, l_ref = MK.attn_fwd64_masked(x64["q"], ke, ve, w.scale, vis)
    go, gl = to_f64(o), to_f64(lse)
    assert max_abs(go, o_ref) <= TOL_O_MAXABS and rel_rms(go, o_ref) <= TOL_O_RELRMS
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(gl), fin)  # rows that see no key: L = -inf on both sides
    assert max_abs(gl[fin], l_ref[fin]) <= TOL_L_MAXABS
    if backward:
        dq_r, dk_r, dv_r = MK.attn_bwd64_masked(x64["q"], ke, ve, x64["do"], w.scale, vis)
        grp = w.H // w.kv_heads
        dk_r = dk_r.reshape(w.B, w.kv_heads, grp, w.N, w.d).sum(axis=2)
        dv_r = dv_r.reshape(w.B, w.kv_heads, grp, w.N, w.d).sum(axis=2)
        for name, a, b in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
            assert np.all(np.isfinite(to_f64(a))), name
            assert rel_rms(to_f64(a), b) <= TOL_GRAD_RELRMS, (name, rel_rms(to_f64(a), b))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(True, 1), (True, 100), (True, 300), (False, 100), (False, 129)])
def test_sliding_window(fa, dtype, d, causal, window):
    _check(fa, Workload("win", 2, 2, 700, d, dtype, causal, "normal", 400 + window + d), window=window)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("heads,density", [(1, 0.5), (3, 0.4), (3, 1.0)])
def test_block_sparse(fa, d, causal, heads, density):
    bm = _block_mask(heads, 640, density, 10 + heads, empty_row=None)
    bm[..., 0] = 1
    _check(fa, Workload("bs", 2, 3, 640, d, "bf16", causal, "normal", 500 + d + heads), bm=bm)


def test_block_mask_window_and_gqa_together(fa):
    bm = _block_mask(4, 1000, 0.6, 21)
    _check(fa, Workload("mix", 1, 4, 1000, 128, "bf16", True, "normal", 600, Hkv=2), window=300, bm=bm)
    _check(fa, Workload("mix", 1, 4, 1000, 64, "fp16", False, "normal", 601, Hkv=1), window=200, bm=bm)


def test_rows_that_see_no_key(fa):
    bm = _block_mask(1, 500, 1.0, 22, empty_row=2)  # query rows 256..383 see nothing
    _check(fa, Workload("empty", 1, 2, 500, 64, "bf16", False, "normal", 700), bm=bm)
    bm2 = _block_mask(1, 500, 1.0, 23)
    bm2[:, :, 1] = 0  # key block 1 seen by nobody: its dK, dV are zero
    _check(fa, Workload("empty", 1, 2, 500, 128, "bf16", True, "normal", 701), bm=bm2)


def test_forward_d256_masked(fa):
    bm = _block_mask(1, 600, 0.5, 24)
    bm[..., 0] = 1
    _check(fa, Workload("m256", 1, 2, 600, 256, "bf16", True, "normal", 702), window=250, bm=bm, backward=False)


@pytest.mark.parametrize("causal,window", [(True, 250), (False, 129)])
def test_d256_masked_forward_backward(fa, causal, window):
    # the d = 256 backward's masked variant: one CTA per (key tile, half of d), step list built
    # from the block mask and the window
    bm = _block_mask(2, 600, 0.6, 25)
    bm[..., 0] = 1
    _check(fa, Workload("m256b", 1, 2, 600, 256, "bf16", causal, "normal", 703 + window), window=window, bm=bm)


def test_visited_tiles_follow_the_nonzero_blocks(fa):
    # Proposition 4: the work is the number of (query tile, key tile) pairs with a visible score
    n, h = 2048, 2
    for causal, window, density in [(False, 0, 0.3), (True, 0, 0.5), (True, 512, 1.0), (False, 300, 0.7)]:
        bm = _block_mask(h, n, density, 30 + window)
        w = Workload("count", 1, h, n, 128, "bf16", causal, "normal", 800)
        x = make_inputs(w, with_do=False)
        dev = {k: to_device(v, w.dtype) for k, v in x.items()}
        fa.fa_tile_counter(reset=True)
        fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=causal, window=window,
                             block_mask=torch.from_numpy(bm).cuda())
        torch.cuda.synchronize()
        assert fa.fa_tile_counter() == MK.blocks_visited(n, causal, window, bm).sum()


def test_long_sequence_sliding_window_sampled_rows(fa):
    # the long-sequence workload (1, 8, 65536, 64, causal) with a 4096-key window: sampled rows
    w = Workload("long_win", 1, 8, 65536, 64, "bf16", True, "normal", 900)
    x = make_inputs(w, with_do=False)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=True, window=4096)
    fa.fa_check_device_error()
    rng = np.random.default_rng(9)
    samples = [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 8, 40), rng.integers(0, 65536, 40))]
    samples += [(0, 0, 0), (0, 7, 65535), (0, 3, 4095), (0, 3, 4096), (0, 5, 4097)]
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    o_ref, l_ref = MK.attn_fwd64_masked_rows(x64["q"], x64["k"], x64["v"], w.scale, samples, True, 4096)
    go, gl = to_f64(o), to_f64(lse)
    got_o = np.stack([go[b, h, i] for b, h, i in samples])
    got_l = np.array([gl[b, h, i] for b, h, i in samples])
    assert max_abs(got_o, o_ref) <= TOL_O_MAXABS and rel_rms(got_o, o_ref) <= TOL_O_RELRMS
    assert max_abs(got_l, l_ref) <= TOL_L_MAXABS
