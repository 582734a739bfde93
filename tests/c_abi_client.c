/*
 * A plain C client of the attention library's C ABI (include/attn.h): no C++, no Python, no PyTorch.
 *
 * It makes seeded inputs (a 32-bit linear congruential generator mapped to [-2, 2), rounded to bf16), allocates
 * its own device buffers with the CUDA runtime, and runs
 *   - one causal GQA prefill through attn_fwd (B=1, Hq=4, Hkv=2, L=200, D=128: a ragged second tile), and
 *   - one GQA decode through attn_decode (B=3, Hq=16, Hkv=4, Lmax=300, D=128, kv_lens 300, 77, 1), and
 *   - one packed causal prefill with rotary embedding through attn_fwd_ex and its parameter struct (two
 *     sequences of 70 and 130 queries over 100 and 130 keys, Hq=4, Hkv=2, D=64, fp32 output, rotated keys
 *     returned in a caller buffer; cos/sin tables of p * 10000^(-2i/D) computed here),
 *   - one multi-token decode through attn_decode_multi (B=2, Hq=8, Hkv=2, Lq=4, Lmax=200, D=128, kv_lens 200, 9),
 *   - one paged decode through attn_decode_paged (B=2, Hq=8, Hkv=2, D=64, 16-key pages in a pool of 12, a
 *     shuffled block table, kv_lens 100, 37),
 * checks the status codes (and that a call with an unsupported head dim is refused before any launch), and
 * writes every input and output as a raw little-endian file into the directory given as argv[1]: the test that
 * builds and runs this program compares the outputs with the fp64 oracle.
 *
 * Exit status 0 on success; otherwise a message on stderr.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "attn.h"

static uint32_t lcg_state = 12345u;

static float next_uniform(void) {
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return (float)(lcg_state >> 8) * (1.0f / 16777216.0f) * 4.0f - 2.0f;
}

/* fp32 -> bf16 bits, round to nearest even (the inputs are finite) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int fail(const char* what, int code) {
  fprintf(stderr, "c_abi_client: %s failed (%d: %s)\n", what, code, attn_status_string(code));
  return 1;
}

static int cuda_ok(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "c_abi_client: %s: %s\n", what, cudaGetErrorString(e));
    return 0;
  }
  return 1;
}

static int write_file(const char* dir, const char* name, const void* data, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (f == NULL) {
    fprintf(stderr, "c_abi_client: cannot write %s\n", path);
    return 0;
  }
  const size_t n = fwrite(data, 1, bytes, f);
  fclose(f);
  return n == bytes;
}

/* a bf16 tensor of n elements: host copy filled from the generator, device copy */
static int make_bf16(size_t n, uint16_t** host, void** dev) {
  *host = (uint16_t*)malloc(n * sizeof(uint16_t));
  if (*host == NULL) return 0;
  for (size_t i = 0; i < n; ++i) (*host)[i] = to_bf16(next_uniform());
  if (!cuda_ok(cudaMalloc(dev, n * sizeof(uint16_t)), "cudaMalloc")) return 0;
  return cuda_ok(cudaMemcpy(*dev, *host, n * sizeof(uint16_t), cudaMemcpyHostToDevice), "cudaMemcpy");
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <output directory>\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  int st;

  /* ---- prefill ---- */
  {
    const int B = 1, Hq = 4, Hkv = 2, L = 200, D = 128;
    const size_t nq = (size_t)B * Hq * L * D, nk = (size_t)B * Hkv * L * D, nl = (size_t)B * Hq * L;
    uint16_t *hq, *hk, *hv;
    void *dq, *dk, *dv, *dout;
    float* dlse;
    if (!make_bf16(nq, &hq, &dq) || !make_bf16(nk, &hk, &dk) || !make_bf16(nk, &hv, &dv)) return 1;
    if (!cuda_ok(cudaMalloc(&dout, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlse, nl * sizeof(float)), "cudaMalloc"))
      return 1;
    /* an unsupported head dim is refused on the host, before any launch */
    st = attn_fwd(dq, dk, dv, dout, dlse, B, Hq, Hkv, L, L, 96, 0.1f, 1, NULL);
    if (st == ATTN_OK) return fail("attn_fwd with D = 96 (should be refused)", st);
    st = attn_fwd(dq, dk, dv, dout, dlse, B, Hq, Hkv, L, L, D, 0.08838834764831845f, 1, NULL);
    if (st != ATTN_OK) return fail("attn_fwd", st);
    st = attn_get_device_status(NULL);
    if (st != ATTN_OK) return fail("attn_get_device_status after attn_fwd", st);
    uint16_t* hout = (uint16_t*)malloc(nq * sizeof(uint16_t));
    float* hlse = (float*)malloc(nl * sizeof(float));
    if (hout == NULL || hlse == NULL) return 1;
    if (!cuda_ok(cudaMemcpy(hout, dout, nq * sizeof(uint16_t), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hlse, dlse, nl * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy"))
      return 1;
    if (!write_file(dir, "prefill_q.bf16", hq, nq * 2) || !write_file(dir, "prefill_k.bf16", hk, nk * 2) ||
        !write_file(dir, "prefill_v.bf16", hv, nk * 2) || !write_file(dir, "prefill_out.bf16", hout, nq * 2) ||
        !write_file(dir, "prefill_lse.f32", hlse, nl * 4))
      return 1;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dlse);
    free(hq); free(hk); free(hv); free(hout); free(hlse);
  }

  /* ---- decode ---- */
  {
    const int B = 3, Hq = 16, Hkv = 4, Lmax = 300, D = 128;
    const int lens[3] = {300, 77, 1};
    const size_t nq = (size_t)B * Hq * D, nc = (size_t)B * Hkv * Lmax * D, nl = (size_t)B * Hq;
    uint16_t *hq, *hk, *hv;
    void *dq, *dk, *dv, *dout;
    int* dlens;
    float* dlse;
    if (!make_bf16(nq, &hq, &dq) || !make_bf16(nc, &hk, &dk) || !make_bf16(nc, &hv, &dv)) return 1;
    if (!cuda_ok(cudaMalloc(&dout, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlse, nl * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlens, sizeof lens), "cudaMalloc") ||
        !cuda_ok(cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice), "cudaMemcpy"))
      return 1;
    st = attn_decode(dq, dk, dv, dlens, dout, dlse, B, Hq, Hkv, Lmax, D, 0.08838834764831845f, NULL);
    if (st != ATTN_OK) return fail("attn_decode", st);
    st = attn_get_device_status(NULL);
    if (st != ATTN_OK) return fail("attn_get_device_status after attn_decode", st);
    uint16_t* hout = (uint16_t*)malloc(nq * sizeof(uint16_t));
    float* hlse = (float*)malloc(nl * sizeof(float));
    if (hout == NULL || hlse == NULL) return 1;
    if (!cuda_ok(cudaMemcpy(hout, dout, nq * sizeof(uint16_t), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hlse, dlse, nl * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy"))
      return 1;
    if (!write_file(dir, "decode_q.bf16", hq, nq * 2) || !write_file(dir, "decode_kc.bf16", hk, nc * 2) ||
        !write_file(dir, "decode_vc.bf16", hv, nc * 2) || !write_file(dir, "decode_lens.i32", lens, sizeof lens) ||
        !write_file(dir, "decode_out.bf16", hout, nq * 2) || !write_file(dir, "decode_lse.f32", hlse, nl * 4))
      return 1;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dlse); cudaFree(dlens);
    free(hq); free(hk); free(hv); free(hout); free(hlse);
  }
  /* ---- packed prefill with RoPE through attn_fwd_ex ---- */
  {
    const int Hq = 4, Hkv = 2, D = 64, maxpos = 160;
    const int cu_q[3] = {0, 70, 200}, cu_k[3] = {0, 100, 230};
    const int total_q = 200, total_k = 230;
    const size_t nq = (size_t)total_q * Hq * D, nk = (size_t)total_k * Hkv * D, nl = (size_t)total_q * Hq;
    const size_t nt = (size_t)maxpos * (D / 2);
    uint16_t *hq, *hk, *hv;
    void *dq, *dk, *dv, *dkout;
    float *dout, *dlse, *dcos, *dsin;
    int *dcuq, *dcuk;
    float* hcos = (float*)malloc(nt * sizeof(float));
    float* hsin = (float*)malloc(nt * sizeof(float));
    if (hcos == NULL || hsin == NULL) return 1;
    for (int p = 0; p < maxpos; ++p)
      for (int i = 0; i < D / 2; ++i) {
        const double a = (double)p * pow(10000.0, -2.0 * i / D);
        hcos[(size_t)p * (D / 2) + i] = (float)cos(a);
        hsin[(size_t)p * (D / 2) + i] = (float)sin(a);
      }
    if (!make_bf16(nq, &hq, &dq) || !make_bf16(nk, &hk, &dk) || !make_bf16(nk, &hv, &dv)) return 1;
    if (!cuda_ok(cudaMalloc((void**)&dout, nq * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlse, nl * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dkout, nk * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dcos, nt * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dsin, nt * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dcuq, sizeof cu_q), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dcuk, sizeof cu_k), "cudaMalloc") ||
        !cuda_ok(cudaMemcpy(dcos, hcos, nt * sizeof(float), cudaMemcpyHostToDevice), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(dsin, hsin, nt * sizeof(float), cudaMemcpyHostToDevice), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(dcuq, cu_q, sizeof cu_q, cudaMemcpyHostToDevice), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(dcuk, cu_k, sizeof cu_k, cudaMemcpyHostToDevice), "cudaMemcpy"))
      return 1;
    attn_fwd_params p;
    memset(&p, 0, sizeof p);
    p.q = dq;
    p.k = dk;
    p.v = dv;
    p.out = dout;
    p.lse = dlse;
    p.B = 2;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = 130;
    p.Lkv = 130;
    p.D = D;
    p.scale = 0.125f;
    p.causal = 1;
    p.out_dtype = ATTN_DTYPE_F32;
    p.cu_seqlens_q = dcuq;
    p.cu_seqlens_k = dcuk;
    p.total_q = total_q;
    p.total_k = total_k;
    p.stream = NULL;
    p.rope.cos = dcos;
    p.rope.sin = dsin;
    p.rope.max_pos = maxpos;
    p.rope.style = ATTN_ROPE_HALF;
    p.rope.k_out = dkout;
    st = attn_fwd_ex(&p);
    if (st != ATTN_OK) return fail("attn_fwd_ex (packed, RoPE)", st);
    st = attn_get_device_status(NULL);
    if (st != ATTN_OK) return fail("attn_get_device_status after attn_fwd_ex", st);
    float* hout = (float*)malloc(nq * sizeof(float));
    float* hlse = (float*)malloc(nl * sizeof(float));
    uint16_t* hkout = (uint16_t*)malloc(nk * sizeof(uint16_t));
    if (hout == NULL || hlse == NULL || hkout == NULL) return 1;
    if (!cuda_ok(cudaMemcpy(hout, dout, nq * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hlse, dlse, nl * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hkout, dkout, nk * sizeof(uint16_t), cudaMemcpyDeviceToHost), "cudaMemcpy"))
      return 1;
    if (!write_file(dir, "rope_q.bf16", hq, nq * 2) || !write_file(dir, "rope_k.bf16", hk, nk * 2) ||
        !write_file(dir, "rope_v.bf16", hv, nk * 2) || !write_file(dir, "rope_cos.f32", hcos, nt * 4) ||
        !write_file(dir, "rope_sin.f32", hsin, nt * 4) || !write_file(dir, "rope_out.f32", hout, nq * 4) ||
        !write_file(dir, "rope_lse.f32", hlse, nl * 4) || !write_file(dir, "rope_kout.bf16", hkout, nk * 2))
      return 1;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dlse); cudaFree(dkout);
    cudaFree(dcos); cudaFree(dsin); cudaFree(dcuq); cudaFree(dcuk);
    free(hq); free(hk); free(hv); free(hout); free(hlse); free(hkout); free(hcos); free(hsin);
  }
  /* ---- multi-token decode through attn_decode_multi ---- */
  {
    const int B = 2, Hq = 8, Hkv = 2, Lq = 4, Lmax = 200, D = 128;
    const int lens[2] = {200, 9};
    const size_t nq = (size_t)B * Hq * Lq * D, nc = (size_t)B * Hkv * Lmax * D, nl = (size_t)B * Hq * Lq;
    uint16_t *hq, *hk, *hv;
    void *dq, *dk, *dv, *dout;
    int* dlens;
    float* dlse;
    if (!make_bf16(nq, &hq, &dq) || !make_bf16(nc, &hk, &dk) || !make_bf16(nc, &hv, &dv)) return 1;
    if (!cuda_ok(cudaMalloc(&dout, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlse, nl * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlens, sizeof lens), "cudaMalloc") ||
        !cuda_ok(cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice), "cudaMemcpy"))
      return 1;
    attn_decode_multi_params p;
    memset(&p, 0, sizeof p);
    p.q = dq;
    p.kcache = dk;
    p.vcache = dv;
    p.kv_lens = dlens;
    p.out = dout;
    p.lse = dlse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = Lq;
    p.Lmax = Lmax;
    p.D = D;
    p.scale = 0.08838834764831845f;
    p.out_dtype = ATTN_DTYPE_BF16;
    st = attn_decode_multi(&p);
    if (st != ATTN_OK) return fail("attn_decode_multi", st);
    st = attn_get_device_status(NULL);
    if (st != ATTN_OK) return fail("attn_get_device_status after attn_decode_multi", st);
    uint16_t* hout = (uint16_t*)malloc(nq * sizeof(uint16_t));
    float* hlse = (float*)malloc(nl * sizeof(float));
    if (hout == NULL || hlse == NULL) return 1;
    if (!cuda_ok(cudaMemcpy(hout, dout, nq * sizeof(uint16_t), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hlse, dlse, nl * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy"))
      return 1;
    if (!write_file(dir, "multi_q.bf16", hq, nq * 2) || !write_file(dir, "multi_kc.bf16", hk, nc * 2) ||
        !write_file(dir, "multi_vc.bf16", hv, nc * 2) || !write_file(dir, "multi_out.bf16", hout, nq * 2) ||
        !write_file(dir, "multi_lse.f32", hlse, nl * 4))
      return 1;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dlse); cudaFree(dlens);
    free(hq); free(hk); free(hv); free(hout); free(hlse);
  }

  /* ---- paged decode through attn_decode_paged ---- */
  {
    const int B = 2, Hq = 8, Hkv = 2, D = 64, ps = 16, max_pages = 8, num_pages = 12;
    const int lens[2] = {100, 37};
    /* sequence 0 uses 7 pages, sequence 1 uses 3; unused entries hold -1 and are never read */
    const int table[16] = {11, 3, 7, 0, 9, 5, 1, -1,
                           6, 10, 2, -1, -1, -1, -1, -1};
    const size_t nq = (size_t)B * Hq * D, npool = (size_t)num_pages * Hkv * ps * D, nl = (size_t)B * Hq;
    uint16_t *hq, *hk, *hv;
    void *dq, *dk, *dv, *dout;
    int *dlens, *dtable;
    float* dlse;
    if (!make_bf16(nq, &hq, &dq) || !make_bf16(npool, &hk, &dk) || !make_bf16(npool, &hv, &dv)) return 1;
    if (!cuda_ok(cudaMalloc(&dout, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlse, nl * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dlens, sizeof lens), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&dtable, sizeof table), "cudaMalloc") ||
        !cuda_ok(cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(dtable, table, sizeof table, cudaMemcpyHostToDevice), "cudaMemcpy"))
      return 1;
    attn_decode_paged_params p;
    memset(&p, 0, sizeof p);
    p.q = dq;
    p.kpages = dk;
    p.vpages = dv;
    p.block_table = dtable;
    p.kv_lens = dlens;
    p.out = dout;
    p.lse = dlse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.page_size = ps;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.scale = 0.125f;
    p.out_dtype = ATTN_DTYPE_BF16;
    st = attn_decode_paged(&p);
    if (st != ATTN_OK) return fail("attn_decode_paged", st);
    st = attn_get_device_status(NULL);
    if (st != ATTN_OK) return fail("attn_get_device_status after attn_decode_paged", st);
    uint16_t* hout = (uint16_t*)malloc(nq * sizeof(uint16_t));
    float* hlse = (float*)malloc(nl * sizeof(float));
    if (hout == NULL || hlse == NULL) return 1;
    if (!cuda_ok(cudaMemcpy(hout, dout, nq * sizeof(uint16_t), cudaMemcpyDeviceToHost), "cudaMemcpy") ||
        !cuda_ok(cudaMemcpy(hlse, dlse, nl * sizeof(float), cudaMemcpyDeviceToHost), "cudaMemcpy"))
      return 1;
    if (!write_file(dir, "paged_q.bf16", hq, nq * 2) || !write_file(dir, "paged_kp.bf16", hk, npool * 2) ||
        !write_file(dir, "paged_vp.bf16", hv, npool * 2) || !write_file(dir, "paged_out.bf16", hout, nq * 2) ||
        !write_file(dir, "paged_lse.f32", hlse, nl * 4))
      return 1;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dlse); cudaFree(dlens); cudaFree(dtable);
    free(hq); free(hk); free(hv); free(hout); free(hlse);
  }
  attn_release_workspace();
  printf("c_abi_client: prefill, decode, packed RoPE prefill, multi-token and paged decode ran through the C ABI\n");
  return 0;
}
