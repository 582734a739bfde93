"""The library used from plain C: tests/c_abi_client.c is compiled with gcc against include/attn.h and the
built library, allocates its own device buffers with the CUDA runtime and calls attn_fwd and attn_decode --
no Python binding, no PyTorch on that path.  Its outputs (written to files with its inputs) are checked
against the fp64 oracle here.  Compiling and linking the client needs no GPU; running it does."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_06_gb300.build import LIB, build
from tests._parity import assert_attn_close

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_client(out_dir):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc is not installed")
    build()
    exe = os.path.join(out_dir, "c_abi_client")
    libdir = os.path.dirname(LIB)
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O2",
           os.path.join(ROOT, "tests", "c_abi_client.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", libdir, "-l:" + os.path.basename(LIB),
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}:{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = compile_client(str(tmp_path))
    assert os.access(exe, os.X_OK)


def _bf16(path, shape):
    raw = np.fromfile(path, dtype=np.uint16)
    return torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).reshape(shape)


def _f32(path, shape):
    return torch.from_numpy(np.fromfile(path, dtype=np.float32).reshape(shape))


@pytest.mark.gpu
def test_c_client_matches_oracle(tmp_path):
    d = str(tmp_path)
    exe = compile_client(d)
    r = subprocess.run([exe, d], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    f = lambda name: os.path.join(d, name)
    # prefill: B=1, Hq=4, Hkv=2, L=200, D=128, causal
    q, k, v = _bf16(f("prefill_q.bf16"), (1, 4, 200, 128)), _bf16(f("prefill_k.bf16"), (1, 2, 200, 128)), \
        _bf16(f("prefill_v.bf16"), (1, 2, 200, 128))
    out, lse = _bf16(f("prefill_out.bf16"), (1, 4, 200, 128)), _f32(f("prefill_lse.f32"), (1, 4, 200))
    O_ref, lse_ref = oracle.attention(q, k, v, 128 ** -0.5, True)
    assert_attn_close(out, lse, O_ref, lse_ref, "C client prefill")
    # decode: B=3, Hq=16, Hkv=4, Lmax=300, D=128
    q = _bf16(f("decode_q.bf16"), (3, 16, 128))
    kc, vc = _bf16(f("decode_kc.bf16"), (3, 4, 300, 128)), _bf16(f("decode_vc.bf16"), (3, 4, 300, 128))
    lens = np.fromfile(f("decode_lens.i32"), dtype=np.int32).tolist()
    assert lens == [300, 77, 1]
    out, lse = _bf16(f("decode_out.bf16"), (3, 16, 128)), _f32(f("decode_lse.f32"), (3, 16))
    O_ref, lse_ref = oracle.decode(q, kc, vc, lens, 128 ** -0.5)
    assert_attn_close(out, lse, O_ref, lse_ref, "C client decode")
    # packed causal prefill with RoPE through attn_fwd_ex: sequences of 70 / 130 queries over 100 / 130 keys,
    # Hq=4, Hkv=2, D=64, fp32 output, scale 0.125, rotated keys returned in k_out
    cu_q, cu_k = [0, 70, 200], [0, 100, 230]
    q, k, v = _bf16(f("rope_q.bf16"), (200, 4, 64)), _bf16(f("rope_k.bf16"), (230, 2, 64)), \
        _bf16(f("rope_v.bf16"), (230, 2, 64))
    cos, sin = _f32(f("rope_cos.f32"), (160, 32)), _f32(f("rope_sin.f32"), (160, 32))
    out, lse = _f32(f("rope_out.f32"), (200, 4, 64)), _f32(f("rope_lse.f32"), (200, 4))
    O_ref, lse_ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.125, True, rope=(cos, sin, "half"))
    assert_attn_close(out, lse, O_ref, lse_ref, "C client packed RoPE prefill")
    # the rotated keys: each sequence's key j at position j, held in bf16 (one bf16 step of slack where fp32
    # and fp64 arithmetic round to different neighbours)
    kout = _bf16(f("rope_kout.bf16"), (230, 2, 64)).double().numpy()
    kd = k.double().numpy()
    for s in range(2):
        a, e = cu_k[s], cu_k[s + 1]
        want = oracle.round_bf16(oracle.rope_rotate(kd[a:e].transpose(1, 0, 2), np.arange(e - a), cos, sin, "half"))
        got = kout[a:e].transpose(1, 0, 2)
        assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 1e-30)
        assert np.mean(got != want) < 1e-2
    # multi-token decode: B=2, Hq=8, Hkv=2, Lq=4, Lmax=200, D=128, kv_lens 200, 9
    q = _bf16(f("multi_q.bf16"), (2, 8, 4, 128))
    kc, vc = _bf16(f("multi_kc.bf16"), (2, 2, 200, 128)), _bf16(f("multi_vc.bf16"), (2, 2, 200, 128))
    out, lse = _bf16(f("multi_out.bf16"), (2, 8, 4, 128)), _f32(f("multi_lse.f32"), (2, 8, 4))
    O_ref, lse_ref = oracle.decode_multi(q, kc, vc, [200, 9], 128 ** -0.5)
    assert_attn_close(out, lse, O_ref, lse_ref, "C client multi-token decode")
    # paged decode: B=2, Hq=8, Hkv=2, D=64, 16-key pages, pool of 12, kv_lens 100, 37; the cache the pages describe
    q = _bf16(f("paged_q.bf16"), (2, 8, 64))
    kp, vp = _bf16(f("paged_kp.bf16"), (12, 2, 16, 64)), _bf16(f("paged_vp.bf16"), (12, 2, 16, 64))
    table = [[11, 3, 7, 0, 9, 5, 1], [6, 10, 2]]
    kc = torch.zeros((2, 2, 112, 64), dtype=torch.bfloat16)
    vc = torch.zeros((2, 2, 112, 64), dtype=torch.bfloat16)
    for b, pages in enumerate(table):
        for i, pg in enumerate(pages):
            kc[b, :, 16 * i:16 * (i + 1)] = kp[pg]
            vc[b, :, 16 * i:16 * (i + 1)] = vp[pg]
    out, lse = _bf16(f("paged_out.bf16"), (2, 8, 64)), _f32(f("paged_lse.f32"), (2, 8))
    O_ref, lse_ref = oracle.decode(q, kc, vc, [100, 37], 0.125)
    assert_attn_close(out, lse, O_ref, lse_ref, "C client paged decode")
