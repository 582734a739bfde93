"""Every entry point on a caller's non-default stream: the work is ordered on that stream only (inputs made on
the default stream are handed over with an event, outputs read after the side stream is joined), and the results
are bitwise those of the same call on the default stream -- the kernels are deterministic (fixed merge orders).
Passing the stream explicitly and taking it from the current-stream context are both exercised."""
import pytest
import torch

from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import make_decode, make_decode_multi, make_prefill

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    AB.load()
    AB.attn_get_device_status()
    yield
    assert AB.attn_get_device_status() == AB.ATTN_OK


def on_side_stream(fn, explicit):
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    if explicit:
        res = fn(side)
    else:
        with torch.cuda.stream(side):
            res = fn(None)
    torch.cuda.current_stream(DEV).wait_stream(side)
    for t in res:
        t.record_stream(side)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("explicit", [True, False])
def test_prefill_on_side_stream(explicit):
    q, k, v = (t.to(DEV) for t in make_prefill(2, 8, 2, 300, 300, 128, seed=501))
    ref = AB.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    got = on_side_stream(lambda s: AB.attn_fwd(q, k, v, causal=True, stream=s), explicit)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


@pytest.mark.parametrize("explicit", [True, False])
def test_decode_on_side_stream(explicit):
    q, kc, vc, lens = (t.to(DEV) for t in make_decode(4, 32, 8, 2048, 128, seed=502, kv_range=(1, 2048)))
    ref = AB.attn_decode(q, kc, vc, lens)
    torch.cuda.synchronize()
    got = on_side_stream(lambda s: AB.attn_decode(q, kc, vc, lens, stream=s), explicit)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


@pytest.mark.parametrize("explicit", [True, False])
def test_decode_multi_on_side_stream(explicit):
    q, kc, vc, _ = make_decode_multi(3, 16, 4, 4, 600, 128, seed=503)
    q, kc, vc = q.to(DEV), kc.to(DEV), vc.to(DEV)
    lens = torch.tensor([600, 130, 9], dtype=torch.int32, device=DEV)
    ref = AB.attn_decode_multi(q, kc, vc, lens)
    torch.cuda.synchronize()
    got = on_side_stream(lambda s: AB.attn_decode_multi(q, kc, vc, lens, stream=s), explicit)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
