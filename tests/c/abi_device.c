/* A plain C99 program that runs flce_fwd_bwd through include/flce.h on device
 * memory it allocates itself with the CUDA runtime.  Usage:
 *   abi_device <dir> <n> <h> <v> <ignore_index> <reduction>
 * reads <dir>/X.bin (bf16 [n,h]), W.bin (bf16 [v,h]), labels.bin (int32 [n]),
 * writes loss.bin, lse.bin, dX.bin, dW.bin, and prints "ok <status>". */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "flce.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes ? bytes : 1);
  size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

#define CHECK(x)                                        \
  do {                                                  \
    if ((x) != cudaSuccess) {                           \
      printf("cuda error at line %d\n", __LINE__);      \
      return 1;                                         \
    }                                                   \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 7) return 2;
  const char* dir = argv[1];
  flce_problem_t p;
  memset(&p, 0, sizeof p);
  p.n = atoll(argv[2]);
  p.h = atoll(argv[3]);
  p.v = atoll(argv[4]);
  p.ignore_index = atoi(argv[5]);
  p.reduction = (flce_reduction_t)atoi(argv[6]);
  const size_t xb = (size_t)p.n * p.h * 2, wb = (size_t)p.v * p.h * 2, lb = (size_t)p.n * 4;
  void* hx = read_file(dir, "X.bin", xb);
  void* hw = read_file(dir, "W.bin", wb);
  void* hl = read_file(dir, "labels.bin", lb);
  if (!hx || !hw || !hl) return 3;
  const size_t ws_bytes = flce_workspace_bytes(&p);
  if (ws_bytes == 0) return 4;
  void *dx_in, *dw_in, *dl, *dloss, *dlse, *ddx, *ddw, *ws;
  CHECK(cudaMalloc(&dx_in, xb));
  CHECK(cudaMalloc(&dw_in, wb));
  CHECK(cudaMalloc(&dl, lb));
  CHECK(cudaMalloc(&dloss, 4));
  CHECK(cudaMalloc(&dlse, (size_t)p.n * 4));
  CHECK(cudaMalloc(&ddx, xb));
  CHECK(cudaMalloc(&ddw, wb));
  CHECK(cudaMalloc(&ws, ws_bytes));
  CHECK(cudaMemcpy(dx_in, hx, xb, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dw_in, hw, wb, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dl, hl, lb, cudaMemcpyHostToDevice));
  flce_status_t st = flce_fwd_bwd(&p, dx_in, dw_in, (const int32_t*)dl, (float*)dloss, (float*)dlse, ddx, ddw, ws,
                                  ws_bytes, NULL);
  if (st != FLCE_OK) {
    printf("call failed: %s\n", flce_status_string(st));
    return 5;
  }
  st = flce_read_device_status(ws, NULL);
  float loss = 0.f;
  float* lse = (float*)malloc((size_t)p.n * 4);
  void* gx = malloc(xb);
  void* gw = malloc(wb);
  CHECK(cudaMemcpy(&loss, dloss, 4, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(lse, dlse, (size_t)p.n * 4, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(gx, ddx, xb, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(gw, ddw, wb, cudaMemcpyDeviceToHost));
  if (write_file(dir, "loss.bin", &loss, 4) || write_file(dir, "lse.bin", lse, (size_t)p.n * 4) ||
      write_file(dir, "dX.bin", gx, xb) || write_file(dir, "dW.bin", gw, wb))
    return 6;
  cudaFree(dx_in);
  cudaFree(dw_in);
  cudaFree(dl);
  cudaFree(dloss);
  cudaFree(dlse);
  cudaFree(ddx);
  cudaFree(ddw);
  cudaFree(ws);
  printf("ok %d\n", (int)st);
  return 0;
}
