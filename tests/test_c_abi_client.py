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
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}:{os.path.join(CUDA, 'lib64')}",
           "-o", exe]
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
