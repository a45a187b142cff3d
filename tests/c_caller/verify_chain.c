/* A plain C99 caller of libspecverify: it owns its device memory through the
 * CUDA runtime, runs one chain verification and prints the results.
 *
 * Usage: verify_chain DIR B K V T
 * DIR holds the inputs as raw little-endian files: Lp.bin (float
 * [B][K+1][V]), Lq.bin (float [B][K][V]), x.bin (int32 [B][K]), ua.bin
 * (float [B][K]), ur.bin (float [B]). Prints one line per batch row:
 * "status accept_len tok_0 ... tok_K". Exit status 0 on success. */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include "specverify.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes ? bytes : 1);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 1) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s DIR B K V T\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int B = atoi(argv[2]), K = atoi(argv[3]), V = atoi(argv[4]);
  const float T = (float)atof(argv[5]);
  const size_t nLp = (size_t)B * (K + 1) * V * sizeof(float), nLq = (size_t)B * K * V * sizeof(float);
  const size_t nx = (size_t)B * K * sizeof(int32_t), nua = (size_t)B * K * sizeof(float), nur = (size_t)B * sizeof(float);
  void* hLp = read_file(dir, "Lp.bin", nLp);
  void* hLq = read_file(dir, "Lq.bin", nLq);
  void* hx = read_file(dir, "x.bin", nx);
  void* hua = read_file(dir, "ua.bin", nua);
  void* hur = read_file(dir, "ur.bin", nur);
  if (!hLp || !hLq || !hx || !hua || !hur) {
    fprintf(stderr, "cannot read the inputs in %s\n", dir);
    return 1;
  }
  void *dLp = to_device(hLp, nLp), *dLq = to_device(hLq, nLq), *dx = to_device(hx, nx);
  void *dua = to_device(hua, nua), *dur = to_device(hur, nur);
  int32_t *dacc = NULL, *dtok = NULL, *dst = NULL;
  void* ws = NULL;
  const size_t wsb = spec_workspace_bytes(B, K, V, SPEC_F32);
  if (!dLp || !dLq || !dx || !dua || !dur || wsb == 0 || cudaMalloc((void**)&dacc, (size_t)B * 4) != cudaSuccess ||
      cudaMalloc((void**)&dtok, (size_t)B * (K + 1) * 4) != cudaSuccess ||
      cudaMalloc((void**)&dst, (size_t)B * 4) != cudaSuccess || cudaMalloc(&ws, wsb) != cudaSuccess) {
    fprintf(stderr, "device allocation failed\n");
    return 1;
  }
  int rc = spec_verify_chain(dLp, dLq, SPEC_F32, (const int32_t*)dx, (const float*)dua, (const float*)dur, T, B, K,
                             V, dacc, dtok, NULL, NULL, NULL, NULL, dst, ws, wsb, NULL);
  if (rc != SPEC_OK) {
    fprintf(stderr, "spec_verify_chain: %s\n", spec_status_string(rc));
    return 1;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    fprintf(stderr, "cudaDeviceSynchronize failed\n");
    return 1;
  }
  int32_t* acc = (int32_t*)malloc((size_t)B * 4);
  int32_t* tok = (int32_t*)malloc((size_t)B * (K + 1) * 4);
  int32_t* st = (int32_t*)malloc((size_t)B * 4);
  if (cudaMemcpy(acc, dacc, (size_t)B * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(tok, dtok, (size_t)B * (K + 1) * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st, dst, (size_t)B * 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
    fprintf(stderr, "copy back failed\n");
    return 1;
  }
  for (int b = 0; b < B; ++b) {
    printf("%d %d", (int)st[b], (int)acc[b]);
    for (int j = 0; j <= K; ++j) printf(" %d", (int)tok[(size_t)b * (K + 1) + j]);
    printf("\n");
  }
  return 0;
}
