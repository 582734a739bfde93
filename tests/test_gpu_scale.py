"""GPU parity for every kind of finite scale: zero, negative and positive.

The scale multiplies the logits before the mask is added ("GPU 学习日报 Day 24：
Operator Fusion" §3.4, standard chain: S = S / sqrt(d) + mask), so a masked key
must drop out whatever the scale: with scale 0 the weights are uniform over the
visible keys, with a negative scale the smallest raw score dominates.  The
shapes put masking on every path that has it: causal diagonals, ragged last
tiles, Lq < Lkv and Lq > Lkv (rows that see nothing), packed sequences, and
multi-token decode (diagonal tiles and the overlapping last tile of an item).
"""
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import make_decode, make_decode_multi, make_prefill, make_varlen, rope_tables
from tests._parity import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SCALES = [0.0, -0.088, 0.37, -1.3]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    AB.load()
    AB.attn_get_device_status()
    yield
    assert AB.attn_get_device_status() == AB.ATTN_OK


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,D,causal", [
    (1, 4, 2, 333, 333, 64, True),
    (1, 4, 2, 333, 333, 128, True),
    (1, 2, 2, 100, 333, 128, True),    # bottom-right offset
    (1, 2, 2, 333, 100, 64, True),     # first rows see no key
    (2, 4, 2, 300, 300, 128, False),   # ragged last tile, no causal mask
])
def test_prefill_any_scale(scale, B, Hq, Hkv, Lq, Lkv, D, causal):
    q, k, v = make_prefill(B, Hq, Hkv, Lq, Lkv, D, seed=500 + Lq + Lkv + D)
    out, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_packed_any_scale(scale, D):
    q, k, v, cu = make_varlen(4, 8, 2, D, seed=510 + D, seqlens=[5, 130, 1, 333])
    out, lse = AB.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), cu.to(DEV), 333, 333, causal=True,
                                  scale=scale)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu.tolist(), cu.tolist(), scale, True)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("scale", [0.0, -0.088])
def test_prefill_rope_any_scale(scale):
    q, k, v = make_prefill(1, 4, 2, 200, 260, 128, seed=520)
    cos, sin = rope_tables(260, 128)
    rope = (cos.to(DEV), sin.to(DEV), "half")
    out, lse = AB.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=scale, rope=rope)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention(q, k, v, scale, True, rope=(cos, sin, "half"))
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lmax,D,lens", [
    (3, 16, 4, 4, 300, 128, [300, 129, 5]),
    (2, 32, 8, 8, 512, 128, [257, 3]),     # kv_len < Lq: early tokens see nothing
    (2, 16, 4, 2, 1000, 64, [1000, 640]),
])
def test_decode_multi_any_scale(scale, B, Hq, Hkv, Lq, Lmax, D, lens):
    q, kc, vc, _ = make_decode_multi(B, Hq, Hkv, Lq, Lmax, D, seed=530 + Lmax + Lq)
    out, lse = AB.attn_decode_multi(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.tensor(lens, dtype=torch.int32).to(DEV),
                                    scale=scale)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, lens, scale)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("scale", SCALES)
def test_decode_any_scale(scale):
    q, kc, vc, lens = make_decode(5, 32, 8, 3000, 128, seed=540, kv_lens=[3000, 1, 0, 777, 2048])
    out, lse = AB.attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), lens.to(DEV), scale=scale)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), scale)
    assert_attn_close(out.cpu(), lse.cpu(), O_ref, lse_ref, f"scale={scale}")
