/*
 * A plain C client of the attention library's C ABI (include/attn.h): no C++, no Python, no PyTorch.
 *
 * It makes seeded inputs (a 32-bit linear congruential generator mapped to [-2, 2), rounded to bf16), allocates
 * its own device buffers with the CUDA runtime, and runs
 *   - one causal GQA prefill through attn_fwd (B=1, Hq=4, Hkv=2, L=200, D=128: a ragged second tile), and
 *   - one GQA decode through attn_decode (B=3, Hq=16, Hkv=4, Lmax=300, D=128, kv_lens 300, 77, 1),
 * checks the status codes (and that a call with an unsupported head dim is refused before any launch), and
 * writes every input and output as a raw little-endian file into the directory given as argv[1]: the test that
 * builds and runs this program compares the outputs with the fp64 oracle.
 *
 * Exit status 0 on success; otherwise a message on stderr.
 */
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
  attn_release_workspace();
  printf("c_abi_client: prefill and decode ran through the C ABI\n");
  return 0;
}
