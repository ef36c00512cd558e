/* uly_c_example.c -- the library driven through its C ABI alone (no Python,
 * no PyTorch): device buffers come from the CUDA runtime, the shard inputs
 * from raw files, and one fused call (uly_sp_attention) writes the output
 * shards back to raw files.
 *
 *   uly_c_example DIR B P S_l R REP_MODE Hq Hkv D N_RANGES
 *
 * reads  DIR/q<p>.bin, DIR/k<p>.bin, DIR/v<p>.bin  (bf16 shards, [B, rows, H, D])
 *        DIR/ranges.bin                           (int32 [B, N_RANGES, 2], if N_RANGES > 0)
 * writes DIR/o<p>.bin                              (bf16 shards, [B, rows, Hq, D])
 * and exits 0 when every call returned ULY_OK. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "uly.h"

static int fail(const char* what, int code) {
  fprintf(stderr, "%s failed: %d\n", what, code);
  return 1;
}

/* Reads exactly `bytes` bytes of DIR/NAME into a new device buffer. */
static void* load(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* host = malloc(bytes ? bytes : 1);
  void* dev = NULL;
  const int ok = host && fread(host, 1, bytes, f) == bytes && fgetc(f) == EOF &&
                 cudaMalloc(&dev, bytes ? bytes : 1) == cudaSuccess &&
                 cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) == cudaSuccess;
  fclose(f);
  free(host);
  if (!ok) {
    if (dev) cudaFree(dev);
    return NULL;
  }
  return dev;
}

static int save(const char* dir, const char* name, const void* dev, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void* host = malloc(bytes ? bytes : 1);
  if (!host || cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
    free(host);
    return 1;
  }
  FILE* f = fopen(path, "wb");
  const int ok = f && fwrite(host, 1, bytes, f) == bytes;
  if (f) fclose(f);
  free(host);
  return ok ? 0 : 1;
}

int main(int argc, char** argv) {
  if (argc != 11) {
    fprintf(stderr, "usage: %s DIR B P S_l R REP_MODE Hq Hkv D N_RANGES\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  uly_desc d;
  memset(&d, 0, sizeof d);
  d.B = atoi(argv[2]);
  d.P = atoi(argv[3]);
  d.S_l = atoi(argv[4]);
  d.R = atoi(argv[5]);
  d.rep_mode = atoi(argv[6]);
  d.Hq = atoi(argv[7]);
  d.Hkv = atoi(argv[8]);
  d.D = atoi(argv[9]);
  d.dtype = ULY_BF16;
  d.masked_rows = ULY_ROWS_SDPA;
  const int n_ranges = atoi(argv[10]);
  if (d.P < 1 || d.P > ULY_MAX_RANKS || n_ranges < 0) return fail("arguments", -1);

  if (cudaSetDevice(0) != cudaSuccess) return fail("cudaSetDevice", -1);
  uly_plan* plan = NULL;
  int rc = uly_plan_create(&d, 0, &plan);
  if (rc != ULY_OK) return fail("uly_plan_create", rc);

  void* q[ULY_MAX_RANKS] = {0};
  void* k[ULY_MAX_RANKS] = {0};
  void* v[ULY_MAX_RANKS] = {0};
  void* o[ULY_MAX_RANKS] = {0};
  size_t o_bytes[ULY_MAX_RANKS] = {0};
  int32_t* ranges = NULL;
  int status = 0;
  for (int p = 0; p < d.P && !status; ++p) {
    const int64_t rq = uly_plan_shard_rows(plan, p, 0), rk = uly_plan_shard_rows(plan, p, 1);
    const size_t qb = (size_t)d.B * (size_t)rq * (size_t)d.Hq * (size_t)d.D * 2;
    const size_t kb = (size_t)d.B * (size_t)rk * (size_t)d.Hkv * (size_t)d.D * 2;
    char name[64];
    snprintf(name, sizeof name, "q%d.bin", p);
    q[p] = load(dir, name, qb);
    snprintf(name, sizeof name, "k%d.bin", p);
    k[p] = load(dir, name, kb);
    snprintf(name, sizeof name, "v%d.bin", p);
    v[p] = load(dir, name, kb);
    o_bytes[p] = qb;
    if (!q[p] || !k[p] || !v[p] || cudaMalloc(&o[p], qb) != cudaSuccess) status = fail("inputs", p);
  }
  if (!status && n_ranges > 0) {
    ranges = (int32_t*)load(dir, "ranges.bin", (size_t)d.B * (size_t)n_ranges * 2 * sizeof(int32_t));
    if (!ranges) status = fail("ranges", -1);
  }
  if (!status) {
    const float scale = (float)(1.0 / sqrt((double)d.D)); /* rounded once, from double */
    rc = uly_sp_attention(plan, (const void* const*)q, (const void* const*)k, (const void* const*)v, NULL, ranges,
                          n_ranges, scale, 0, NULL, NULL, NULL, o, NULL, NULL);
    if (rc != ULY_OK) status = fail("uly_sp_attention", rc);
  }
  if (!status) {
    rc = uly_sync_status(plan, NULL);
    if (rc != ULY_OK) status = fail(uly_status_string(rc), rc);
  }
  for (int p = 0; p < d.P && !status; ++p) {
    char name[64];
    snprintf(name, sizeof name, "o%d.bin", p);
    if (save(dir, name, o[p], o_bytes[p])) status = fail("outputs", p);
  }
  for (int p = 0; p < d.P; ++p) {
    cudaFree(q[p]);
    cudaFree(k[p]);
    cudaFree(v[p]);
    cudaFree(o[p]);
  }
  cudaFree(ranges);
  uly_plan_destroy(plan);
  return status;
}
