"""GPU parity of split-KV decode (attn_decode) against the fp64 oracle.

Inputs are the same seeded bf16 tensors on both sides.  Small cases cover
every grouped-head width the kernel specialises (1, 2, 4, 8 and a grouping
that needs several head groups), both head dims, ragged and degenerate
lengths (0, 1, not a multiple of the stage or the chunk, == Lmax) and several
minimum slice sizes (down to one key per CTA, which splits rows into many
partials); the two decode workloads run at full size with every row checked
(the 8 x 4096 cache and the 32k-128k-key caches), and a 2^20-key cache on
sampled heads.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300 import binding as AB
from attention_attn_fwd_06_gb300.build import build
from attention_attn_fwd_06_gb300.inputs import WORKLOADS, make_decode, make_pages
from tests._parity import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    AB.load()
    AB.attn_get_device_status()


def run(q, kc, vc, lens, scale, chunk=0, out_dtype=torch.bfloat16):
    dev = torch.device("cuda:0")
    out, lse = AB.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), lens.to(dev), scale=scale, chunk=chunk,
                              out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D,lens", [
    (2, 4, 4, 300, 128, [300, 17]),        # MHA (1 head per kv head)
    (2, 8, 4, 200, 128, [1, 199]),         # 2 heads per kv head
    (3, 16, 4, 513, 128, [513, 64, 65]),   # 4 heads (the decode workload's grouping)
    (2, 16, 2, 257, 128, [257, 128]),      # 8 heads
    (1, 32, 2, 130, 128, [130]),           # 16 heads -> two head groups of 8
    (2, 12, 4, 100, 128, [100, 3]),        # 3 heads -> three groups of 1
    (2, 8, 8, 333, 64, [333, 129]),        # D = 64, MHA
    (2, 16, 4, 400, 64, [255, 400]),       # D = 64, 4 heads
    (1, 16, 2, 77, 64, [77]),              # D = 64, 8 heads
])
def test_decode_small(B, Hq, Hkv, Lmax, D, lens):
    q, kc, vc, _ = make_decode(B, Hq, Hkv, Lmax, D, seed=7 + Lmax)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    scale = D ** -0.5
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale)
    # chunk = smallest key slice per CTA: 1 and 7 split rows into many partials (stresses the merge)
    for chunk in (0, 1, 7, 64, 192):
        O, lse = run(q, kc, vc, lens_t, scale, chunk=chunk)
        assert_attn_close(O, lse, O_ref, lse_ref, f"chunk={chunk}")


def test_decode_tiny_lengths_many_rows():
    # Rows with one to three keys: one CTA per row, not one CTA walking them all.
    lens = [1, 2, 3, 1, 1, 2, 3, 3, 2, 1, 1, 1, 2, 2, 3, 1]
    q, kc, vc, _ = make_decode(len(lens), 32, 8, 8, 128, seed=5)
    for chunk in (0, 64):
        O, lse = run(q, kc, vc, torch.tensor(lens, dtype=torch.int32), 0.088, chunk=chunk)
        O_ref, lse_ref = oracle.decode(q, kc, vc, lens, 0.088)
        assert_attn_close(O, lse, O_ref, lse_ref, f"chunk={chunk}")


@pytest.mark.parametrize("B,Hq,Hkv", [
    (40, 16, 4),   # more sequences than a warp has lanes: the length walk and the row search take two passes
    (70, 16, 2),   # 8 heads per kv head: more sequences than the shared-memory length cache holds
])
def test_decode_many_sequences(B, Hq, Hkv):
    g = torch.Generator().manual_seed(B)
    lens = torch.randint(0, 300, (B,), generator=g, dtype=torch.int32)
    lens[3] = 0  # an empty sequence among them
    q, kc, vc, _ = make_decode(B, Hq, Hkv, 300, 128, seed=50 + B)
    for chunk in (0, 7):
        O, lse = run(q, kc, vc, lens, 0.088, chunk=chunk)
        O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), 0.088)
        assert_attn_close(O, lse, O_ref, lse_ref, f"B={B} chunk={chunk}")


def test_decode_all_sequences_empty():
    q, kc, vc, _ = make_decode(2, 8, 2, 64, 128, seed=4)
    O, lse = run(q, kc, vc, torch.zeros(2, dtype=torch.int32), 0.088)
    assert torch.all(O == 0) and torch.all(torch.isneginf(lse))


def test_decode_zero_length_rows():
    q, kc, vc, _ = make_decode(3, 8, 2, 96, 128, seed=3)
    lens = torch.tensor([0, 96, 0], dtype=torch.int32)
    O, lse = run(q, kc, vc, lens, 0.088)
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), 0.088)
    assert torch.all(O[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_never_reads_past_kv_len():
    # Cache rows at or beyond kv_len hold NaN: any read of them would poison O.
    q, kc, vc, _ = make_decode(2, 8, 2, 640, 128, seed=11)
    lens = [300, 577]
    for b, n in enumerate(lens):
        kc[b, :, n:] = float("nan")
        vc[b, :, n:] = float("nan")
    O, lse = run(q, kc, vc, torch.tensor(lens, dtype=torch.int32), 0.09, chunk=128)
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, 0.09)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_fp32_output_and_scale():
    q, kc, vc, _ = make_decode(2, 8, 2, 200, 128, seed=5)
    lens = torch.tensor([200, 150], dtype=torch.int32)
    O, lse = run(q, kc, vc, lens, 0.5, out_dtype=torch.float32)
    assert O.dtype == torch.float32
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), 0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_peaked_logits_rescale():
    # Large logits make the running max rise often, exercising the O rescale.
    q, kc, vc, _ = make_decode(2, 16, 4, 1024, 128, seed=13)
    q = (q.float() * 8).to(torch.bfloat16)
    kc[:, :, 700:710] = (kc[:, :, 700:710].float() * 4).to(torch.bfloat16)
    lens = torch.tensor([1024, 901], dtype=torch.int32)
    O, lse = run(q, kc, vc, lens, 128 ** -0.5, chunk=256)
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), 128 ** -0.5)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_deterministic():
    q, kc, vc, lens = make_decode(2, 16, 4, 2048, 128, seed=17, kv_range=(1, 2048))
    a = run(q, kc, vc, lens, 0.088)
    b = run(q, kc, vc, lens, 0.088)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_out_of_range_length_is_flagged():
    q, kc, vc, _ = make_decode(2, 8, 2, 128, 128, seed=19)
    lens = torch.tensor([128, 500], dtype=torch.int32)  # 500 > Lmax: clamped to 128, flagged
    O, lse = run(q, kc, vc, lens, 0.088)
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_BOUNDS
    assert AB.attn_get_device_status() == AB.ATTN_OK  # reading clears it
    O_ref, lse_ref = oracle.decode(q, kc, vc, [128, 128], 0.088)
    assert_attn_close(O, lse, O_ref, lse_ref)


def test_decode_matches_last_row_of_causal_prefill_oracle():
    # Same data through decode; the oracle's decode is pinned to causal prefill's last row.
    q, kc, vc, _ = make_decode(1, 8, 2, 256, 128, seed=23)
    O, lse = run(q, kc, vc, torch.tensor([256], dtype=torch.int32), 0.088)
    qp = torch.zeros(1, 8, 256, 128, dtype=torch.bfloat16)
    qp[0, :, 255] = q[0]
    Op, lsep = oracle.attention(qp, kc, vc, 0.088, True)
    assert_attn_close(O[0], lse[0], Op[0, :, 255], lsep[0, :, 255])


def test_decode_workload_gqa_full():
    w = WORKLOADS["decode_gqa"]
    q, kc, vc, lens = make_decode(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed, kv_range=w.kv_range)
    O, lse = run(q, kc, vc, lens, w.scale)
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), w.scale)
    assert_attn_close(O, lse, O_ref, lse_ref, "decode_gqa")
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_decode_workload_long_full():
    # The long-context workload (kv_len 32k / 64k / 96k / 128k, every row split over many CTAs and merged through the
    # partials): every (sequence, query head) row against the oracle, element by element.
    w = WORKLOADS["decode_long"]
    q, kc, vc, lens = make_decode(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed, kv_lens=w.kv_lens)
    O, lse = run(q, kc, vc, lens, w.scale)
    assert torch.isfinite(O).all() and torch.isfinite(lse).all()
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), w.scale)
    assert_attn_close(O, lse, O_ref, lse_ref, "decode_long")
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_decode_million_key_cache_sampled():
    """A 2^20-key cache (8x the longest workload): one sequence filling it, one of 777,777 keys; sampled heads of
    both against the oracle."""
    B, Hq, Hkv, Lmax, D = 2, 8, 2, 1 << 20, 128
    q, kc, vc, lens = make_decode(B, Hq, Hkv, Lmax, D, seed=1 << 20, kv_lens=[Lmax, 777_777])
    O, lse = run(q, kc, vc, lens, D ** -0.5)
    assert torch.isfinite(O).all() and torch.isfinite(lse).all()
    assert AB.attn_get_device_status() == AB.ATTN_OK
    heads = [(0, 0), (0, 5), (1, 3), (1, 7)]
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), D ** -0.5, heads=heads)
    bi = np.array([b for b, _ in heads])
    hi = np.array([h for _, h in heads])
    assert_attn_close(O[torch.as_tensor(bi), torch.as_tensor(hi)], lse[torch.as_tensor(bi), torch.as_tensor(hi)],
                      O_ref[bi, hi], lse_ref[bi, hi], "2^20-key decode")


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D,page_size", [
    (3, 16, 4, 700, 128, 16),    # vLLM-sized pages, 4 heads per kv head
    (3, 16, 4, 700, 128, 48),    # a page size that is not a power of two
    (2, 32, 8, 1000, 128, 256),  # pages longer than a pipeline stage
    (2, 8, 8, 333, 64, 32),      # D = 64, MHA
    (1, 16, 2, 129, 128, 8),     # smallest page size, 8 heads per kv head
])
def test_decode_paged_matches_contiguous_and_oracle(B, Hq, Hkv, Lmax, D, page_size):
    q, kc, vc, lens = make_decode(B, Hq, Hkv, Lmax, D, seed=900 + page_size, kv_range=(1, Lmax))
    kp, vp, table = make_pages(kc, vc, page_size, seed=901)
    # entries past a sequence's last page hold -1, as serving engines pad block tables: never read, never flagged
    for b in range(B):
        table[b, (int(lens[b]) + page_size - 1) // page_size:] = -1
    AB.attn_get_device_status()
    dev = torch.device("cuda:0")
    scale = D ** -0.5
    for chunk in (0, 7):
        Oc, lc = AB.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), lens.to(dev), scale=scale, chunk=chunk)
        Op, lp = AB.attn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lens.to(dev), scale=scale,
                                      chunk=chunk)
        torch.cuda.synchronize()
        # same keys in the same stages: the paged result is bitwise the contiguous one
        assert torch.equal(Op.cpu(), Oc.cpu()) and torch.equal(lp.cpu(), lc.cpu())
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), scale)
    assert_attn_close(Op.cpu(), lp.cpu(), O_ref, lse_ref)
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_decode_paged_bad_page_id_is_flagged():
    q, kc, vc, lens = make_decode(2, 8, 2, 64, 128, seed=77, kv_lens=[64, 50])
    kp, vp, table = make_pages(kc, vc, 16, seed=78, fill_unused=0.0)
    table[1, 2] = kp.shape[0] + 5  # outside the pool, on a page that holds keys 32..47 of sequence 1
    dev = torch.device("cuda:0")
    AB.attn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lens.to(dev))
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_BOUNDS
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_device_timeout_is_reported_and_context_survives():
    # The bounded wait every pipeline stage uses, run out on purpose (a barrier nothing arrives on, 2 ms limit):
    # the status word reports the timeout, and the next call works normally.
    AB.attn_get_device_status()
    AB.attn_selftest_wait_timeout(2000)
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_TIMEOUT
    assert AB.attn_get_device_status() == AB.ATTN_OK  # read-and-clear
    q, kc, vc, _ = make_decode(2, 8, 2, 300, 128, seed=9)
    lens = [300, 120]
    O, lse = run(q, kc, vc, torch.tensor(lens, dtype=torch.int32), 0.088)
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, 0.088)
    assert_attn_close(O, lse, O_ref, lse_ref)
    assert AB.attn_get_device_status() == AB.ATTN_OK


def test_fault_injection_skip_arrive_times_out_and_recovers(monkeypatch):
    # ATTN_FAULT_INJECT=skip_arrive: CTA 0 withholds one pipeline-slot release, its producer's bounded wait runs
    # out (about a second), the status word reports the timeout, and the next clean call is correct.
    w = WORKLOADS["decode_gqa"]
    q, kc, vc, lens = make_decode(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed, kv_range=w.kv_range)
    AB.attn_get_device_status()
    monkeypatch.setenv("ATTN_FAULT_INJECT", "skip_arrive")
    run(q, kc, vc, lens, w.scale)
    assert AB.attn_get_device_status() == AB.ATTN_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("ATTN_FAULT_INJECT")
    O, lse = run(q, kc, vc, lens, w.scale)
    assert AB.attn_get_device_status() == AB.ATTN_OK
    heads = [(b, h) for b in range(w.B) for h in (0, 31)]
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens.tolist(), w.scale, heads=heads)
    idx_b = [b for b, _ in heads]
    idx_h = [h for _, h in heads]
    assert_attn_close(O[idx_b, idx_h], lse[idx_b, idx_h], O_ref[idx_b, idx_h], lse_ref[idx_b, idx_h])
