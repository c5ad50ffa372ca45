"""Split-KV decode through the C ABI vs the fp64 oracle (attention over the whole cache)."""

import numpy as np
import pytest

from oracle import decode as DEC
from exact_tiled_attention_07_gb300.inputs import DECODE_WORKLOADS, make_decode_inputs, round_to_dtype, to_float64
from helpers import TOL_FP32, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, max_abs, rel_rms, to_device, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _inputs(b, h, hkv, nq, nk, d, dtype, seed, offsets=False):
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((b, h, nq, d), dtype=np.float32)
    k = rng.standard_normal((b, hkv, nk, d), dtype=np.float32)
    v = rng.standard_normal((b, hkv, nk, d), dtype=np.float32)
    if offsets:  # per-key score offsets N(0, 4), as in the long-sequence workload
        q[..., 0] = 1.0
        k[..., 0] = rng.standard_normal((b, hkv, nk), dtype=np.float32) * 2.0 * np.float32(np.sqrt(d))
    return {nm: round_to_dtype(a, dtype) for nm, a in (("q", q), ("k", k), ("v", v))}


def _check(fa, b, h, hkv, nq, nk, d, dtype, splits, seed, offsets=False):
    x = _inputs(b, h, hkv, nq, nk, d, dtype, seed, offsets)
    dev = {k: to_device(v, dtype) for k, v in x.items()}
    o, lse = fa.attention_decode(dev["q"], dev["k"], dev["v"], splits=splits)
    fa.fa_check_device_error()
    x64 = {k: to_float64(v, dtype) for k, v in x.items()}
    o_ref, l_ref = DEC.decode_fwd64(x64["q"], x64["k"], x64["v"], d ** -0.5)
    go, gl = to_f64(o), to_f64(lse)
    if dtype == "fp32":
        assert max_abs(go, o_ref) <= TOL_FP32 and max_abs(gl, l_ref) <= TOL_FP32
    else:
        assert max_abs(go, o_ref) <= TOL_O_MAXABS and rel_rms(go, o_ref) <= TOL_O_RELRMS
        assert max_abs(gl, l_ref) <= TOL_L_MAXABS


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_shapes(fa, dtype, d, splits):
    _check(fa, 2, 8, 2, 1, 1000, d, dtype, splits, 100 + d + splits)


@pytest.mark.parametrize("h,hkv,nq,nk", [(4, 4, 1, 1), (4, 1, 3, 33), (16, 2, 2, 4097), (8, 8, 9, 300),
                                         (32, 4, 1, 20000)])
def test_decode_groups_rows_and_cache_lengths(fa, h, hkv, nq, nk):
    _check(fa, 1, h, hkv, nq, nk, 128, "bf16", 0, 200 + nk)


def test_decode_many_splits_and_score_offsets(fa):
    _check(fa, 2, 8, 8, 1, 3000, 128, "bf16", 64, 300, offsets=True)
    _check(fa, 1, 4, 2, 1, 50, 64, "bf16", 50, 301)  # one key per split


def test_decode_workspace_rules(fa):
    assert fa.fa_decode_workspace_size(1, 8, 2, 1, 100, 128, 1) == 0
    assert fa.fa_decode_workspace_size(1, 8, 2, 1, 100, 128, 4) == 8 * 4 * 129 * 4
    assert fa.fa_decode_workspace_size(1, 8, 2, 1, 3, 128, 10) == 8 * 3 * 129 * 4  # capped at Nk
    q = torch.zeros((1, 8, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 2, 100, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((1, 8, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError, match="workspace"):
        fa.fa_decode(q, k, k, o, lse, 0.1, splits=4, workspace=None)


@pytest.mark.parametrize("h,hkv,nq,nk,splits", [(64, 1, 3, 1000, 0), (8, 2, 40, 300, 0), (8, 2, 40, 300, 2),
                                                (16, 16, 1, 300, 10), (4, 1, 64, 129, 0), (8, 1, 5, 700, 0),
                                                (16, 2, 8, 1000, 3), (8, 8, 1, 129, 2)])
def test_decode_row_tiles_and_empty_pieces(fa, h, hkv, nq, nk, splits):
    # group x Nq above 128 rows (several row tiles per key/value head), 33..64 rows (two
    # copies of the rows on the tensor-core path) and <= 32 rows (four copies); more pieces
    # than key tiles (empty pieces); a one-key last tile, alone in its piece, so that three
    # of the four row copies see no key there
    _check(fa, 2, h, hkv, nq, nk, 128, "bf16", splits, 400 + h + nq)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("nq", [1, 5, 20])
def test_decode_row_copies_per_head_dim(fa, d, nq):
    # 8 query heads on one key/value head: 8, 40 and 160 rows
    _check(fa, 1, 8, 1, nq, 777, d, "fp16", 0, 700 + d + nq)


def test_decode_visits_every_key_tile_once_per_row_tile(fa):
    b, h, hkv, nq, nk, d = 2, 16, 4, 2, 1000, 64
    x = _inputs(b, h, hkv, nq, nk, d, "bf16", 500)
    dev = {k: to_device(v, "bf16") for k, v in x.items()}
    fa.fa_tile_counter(reset=True)
    fa.attention_decode(dev["q"], dev["k"], dev["v"], splits=3)
    torch.cuda.synchronize()
    rows = (h // hkv) * nq
    assert fa.fa_tile_counter() == b * hkv * ((rows + 127) // 128) * ((nk + 127) // 128)


def test_decode_long_cache_sampled_heads(fa):
    # the decode step the benchmark times (B 8, H 32, Hkv 8, Nk 32768, d 128), in the launch
    # configuration it uses, checked on sampled heads against attention over the whole cache
    w = DECODE_WORKLOADS["decode_gqa_bf16"]
    b, h, hkv, nq, nk, d = w.B, w.H, w.Hkv, w.Nq, w.Nk, w.d
    x = make_decode_inputs(w)
    dev = {k: to_device(v, "bf16") for k, v in x.items()}
    o, lse = fa.attention_decode(dev["q"], dev["k"], dev["v"])
    fa.fa_check_device_error()
    go, gl = to_f64(o), to_f64(lse)
    group = h // hkv
    for bi, hi in [(0, 0), (0, 31), (3, 9), (7, 20), (5, 4)]:
        kv = hi // group
        o_ref, l_ref = DEC.decode_fwd64(to_float64(x["q"][bi:bi + 1, hi:hi + 1], "bf16"),
                                        to_float64(x["k"][bi:bi + 1, kv:kv + 1], "bf16"),
                                        to_float64(x["v"][bi:bi + 1, kv:kv + 1], "bf16"), d ** -0.5)
        assert max_abs(go[bi, hi], o_ref[0, 0]) <= TOL_O_MAXABS
        assert rel_rms(go[bi, hi], o_ref[0, 0]) <= TOL_O_RELRMS
        assert max_abs(gl[bi, hi], l_ref[0, 0]) <= TOL_L_MAXABS
