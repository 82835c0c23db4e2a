/* A C caller of libgqa_decode.so: device buffers from cudaMalloc, the workspace sized by
 * gqa_workspace_size, one gqa_decode step, the output copied back.  Used by
 * tests/test_gpu_c_caller.py, which writes the inputs and checks the output.
 *
 * usage: decode_from_c <dir> B T_q S_kv h_q h_kv d_head scale
 *   reads <dir>/q.bin (B*T_q*h_q*d_head f16), k.bin and v.bin (B*S_kv*h_kv*d_head f16),
 *   writes <dir>/o.bin (B*T_q*h_q*d_head f16); exit status 0 on success. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "gqa_decode.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

int main(int argc, char** argv) {
  if (argc != 9) {
    fprintf(stderr, "usage: %s dir B T_q S_kv h_q h_kv d_head scale\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int B = atoi(argv[2]), T_q = atoi(argv[3]), h_q = atoi(argv[5]), h_kv = atoi(argv[6]), D = atoi(argv[7]);
  const int64_t S = atoll(argv[4]);
  const float scale = (float)atof(argv[8]);
  const size_t qb = (size_t)B * T_q * h_q * D * 2, kb = (size_t)B * S * h_kv * D * 2;
  void *hq = read_file(dir, "q.bin", qb), *hk = read_file(dir, "k.bin", kb), *hv = read_file(dir, "v.bin", kb);
  if (!hq || !hk || !hv) {
    fprintf(stderr, "cannot read the inputs\n");
    return 3;
  }
  const size_t ws_bytes = gqa_workspace_size(B, T_q, S, h_q, h_kv, D);
  if (ws_bytes == 0) {
    fprintf(stderr, "gqa_workspace_size: invalid shape or no device\n");
    return 4;
  }
  void *q, *k, *v, *o, *ws;
  if (cudaMalloc(&q, qb) || cudaMalloc(&k, kb) || cudaMalloc(&v, kb) || cudaMalloc(&o, qb) ||
      cudaMalloc(&ws, ws_bytes))
    return 5;
  cudaMemcpy(q, hq, qb, cudaMemcpyHostToDevice);
  cudaMemcpy(k, hk, kb, cudaMemcpyHostToDevice);
  cudaMemcpy(v, hv, kb, cudaMemcpyHostToDevice);
  cudaStream_t st;
  cudaStreamCreate(&st);
  if (gqa_workspace_init(ws, ws_bytes, st) != GQA_OK) return 6;
  gqa_status s = gqa_decode((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, (uint16_t*)o, B, T_q, S, h_q,
                            h_kv, D, scale, ws, ws_bytes, st);
  if (s != GQA_OK) {
    fprintf(stderr, "gqa_decode: %s\n", gqa_status_string(s));
    return 7;
  }
  s = gqa_workspace_check(ws, st);   /* synchronises the stream */
  if (s != GQA_OK) {
    fprintf(stderr, "device status: %s\n", gqa_status_string(s));
    return 8;
  }
  void* ho = malloc(qb);
  if (!ho || cudaMemcpy(ho, o, qb, cudaMemcpyDeviceToHost) != cudaSuccess) return 9;
  char path[4096];
  snprintf(path, sizeof(path), "%s/o.bin", dir);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(ho, 1, qb, f) != qb) return 10;
  fclose(f);
  cudaFree(q);
  cudaFree(k);
  cudaFree(v);
  cudaFree(o);
  cudaFree(ws);
  cudaStreamDestroy(st);
  printf("ok %zu workspace bytes\n", ws_bytes);
  return 0;
}
