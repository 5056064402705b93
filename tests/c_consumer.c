/* A plain C caller of the library's C boundary (include/sp_fused.h): allocates device buffers with
 * the CUDA runtime, fills them from a small host problem, calls sp_fused_reduce_norm on a stream
 * and prints the outputs as hex, one value per line, for the test to compare with the oracle.
 * Usage: c_consumer <input file> <output file>; the input file holds, in this order, as raw
 * little-endian bytes: int32 tp, T_pad, T_valid, H, mode; float eps, scale; then bf16 partials
 * [tp][T_pad][H], residual [T_pad][H], weight [H], bias [H]. Without a GPU it only checks the
 * host-side helpers and exits 0. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "sp_fused.h"

#define CHECK(x)                                                     \
  do {                                                               \
    if ((x) != cudaSuccess) {                                        \
      fprintf(stderr, "CUDA error at %s:%d\n", __FILE__, __LINE__);  \
      return 2;                                                      \
    }                                                                \
  } while (0)

static void* read_all(FILE* f, size_t n) {
  void* p = malloc(n ? n : 1);
  if (p && n && fread(p, 1, n, f) != n) {
    free(p);
    return NULL;
  }
  return p;
}

int main(int argc, char** argv) {
  if (sp_pad_tokens(3500, 16) != 3504 || sp_out_bytes(8, 64, SP_QUANT_NVFP4) != 8 * 32) return 3;
  int count = 0;
  if (argc < 3 || cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    printf("host-only checks passed\n");
    return 0;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 4;
  int32_t hdr[5];
  float fl[2];
  if (fread(hdr, 4, 5, in) != 5 || fread(fl, 4, 2, in) != 2) return 4;
  const int tp = hdr[0], mode = hdr[4];
  const int64_t T_pad = hdr[1], T_valid = hdr[2], H = hdr[3];
  const size_t plane = (size_t)T_pad * H * 2;
  void* h_part = read_all(in, plane * tp);
  void* h_res = read_all(in, plane);
  void* h_w = read_all(in, (size_t)H * 2);
  void* h_b = read_all(in, (size_t)H * 2);
  fclose(in);
  if (!h_part || !h_res || !h_w || !h_b) return 4;
  const int64_t ob = sp_out_bytes(T_pad, H, mode), sb = sp_out_scales_bytes(T_pad, H, mode);
  void *d_part, *d_res, *d_w, *d_b, *d_out, *d_res_out, *d_sc = NULL;
  float* d_scale = NULL;
  CHECK(cudaMalloc(&d_part, plane * tp));
  CHECK(cudaMalloc(&d_res, plane));
  CHECK(cudaMalloc(&d_w, (size_t)H * 2));
  CHECK(cudaMalloc(&d_b, (size_t)H * 2));
  CHECK(cudaMalloc(&d_out, (size_t)ob));
  CHECK(cudaMalloc(&d_res_out, plane));
  if (sb) CHECK(cudaMalloc(&d_sc, (size_t)sb));
  CHECK(cudaMalloc((void**)&d_scale, 4));
  CHECK(cudaMemcpy(d_part, h_part, plane * tp, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_res, h_res, plane, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_w, h_w, (size_t)H * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_b, h_b, (size_t)H * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_scale, &fl[1], 4, cudaMemcpyHostToDevice));
  cudaStream_t s;
  CHECK(cudaStreamCreate(&s));
  const int needs_scale = mode == SP_QUANT_FP8_STATIC || mode == SP_QUANT_NVFP4;
  sp_status st = sp_fused_reduce_norm(d_part, tp, T_pad, T_valid, H, d_res, d_w, d_b, fl[0], mode,
                                      needs_scale ? d_scale : NULL, d_out, d_sc, d_res_out, s);
  if (st != SP_OK) {
    fprintf(stderr, "sp_fused_reduce_norm: %s\n", sp_status_string(st));
    return 5;
  }
  CHECK(cudaStreamSynchronize(s));
  unsigned char* h_out = (unsigned char*)malloc((size_t)ob);
  unsigned char* h_sc = (unsigned char*)malloc(sb ? (size_t)sb : 1);
  unsigned char* h_ro = (unsigned char*)malloc(plane);
  CHECK(cudaMemcpy(h_out, d_out, (size_t)ob, cudaMemcpyDeviceToHost));
  if (sb) CHECK(cudaMemcpy(h_sc, d_sc, (size_t)sb, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(h_ro, d_res_out, plane, cudaMemcpyDeviceToHost));
  FILE* out = fopen(argv[2], "wb");
  if (!out) return 6;
  fwrite(h_out, 1, (size_t)ob, out);
  if (sb) fwrite(h_sc, 1, (size_t)sb, out);
  fwrite(h_ro, 1, plane, out);
  fclose(out);
  printf("device call ok\n");
  return 0;
}
