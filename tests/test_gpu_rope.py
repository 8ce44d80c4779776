"""RoPE kernel vs the oracle's fp64 rotate-half RoPE (within one bf16 ulp)."""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("L,H,d,theta,yarn,orig", [
    (1024, 4, 64, 1e4, 1.0, 0),
    (4096, 2, 128, 1e4, 1.0, 0),
    (8192, 2, 128, 5e5, 32.0, 256),
    (131072, 1, 128, 1e4, 1.0, 0),
])
@pytest.mark.parametrize("transpose", [False, True])
def test_rope_matches_oracle(L, H, d, theta, yarn, orig, transpose):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    x = synth.normal_bf16(77, (L, H, d))
    p = vs.make_params(L, H, H, d, rope_theta=theta, yarn_factor=yarn, yarn_orig_len=orig)
    xt = to_dev(x, dev)
    y = torch.empty_like(xt)
    vs.vs_rope(p, H, xt, y, transpose)
    torch.cuda.synchronize()
    got = f64(bf16_bits_of(y))
    ref = oracle.rope(f64(x), theta, transpose=transpose, yarn_factor=yarn, yarn_orig_len=orig)
    # bf16 spacing at the exact value, plus the fp32 arithmetic error of the
    # kernel (a few fp32 ulps of the inputs' magnitude)
    spacing = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    xin = np.abs(f64(x))
    mag = np.concatenate([xin[..., d // 2:], xin[..., :d // 2]], axis=-1) + xin
    allowed = spacing + 2e-6 * mag * oracle.rope_mscale(yarn)
    assert (np.abs(got - ref) <= allowed).all()
    # the bf16 value is the nearest one except where fp32 rounding lands on a tie
    assert (np.abs(got - oracle.bf16_round(ref)) > 0).mean() < 1e-3


def test_rope_in_place_and_roundtrip():
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    L, H, d = 2048, 3, 64
    x = synth.normal_bf16(78, (L, H, d))
    p = vs.make_params(L, H, H, d)
    xt = to_dev(x, dev)
    y = xt.clone()
    vs.vs_rope(p, H, y, y, False)
    vs.vs_rope(p, H, y, y, True)
    torch.cuda.synchronize()
    assert (y.float() - xt.float()).abs().max().item() <= 0.04
