/*
 * A plain C client of libspanla: no Python, no PyTorch.  It reads a packed
 * pass (metadata and bf16 q, k, v as raw little-endian arrays) from a file,
 * runs span_la_pass, span_la_softmax_pass and span_la_branches_from_state on
 * the current CUDA device through the C ABI of include/spanla.h, and writes
 * the three outputs and the view states back to a file.
 *
 *   spanla_client <input> <output>
 *
 * input:  int32 T, H, V, B; int32 view_cu[V+1]; int32 branch_cu[B+1];
 *         int32 branch_parent[B]; uint16 q[T*H*64], k[...], v[...] (bf16 bits)
 * output: uint16 out_pass[T*H*64]; float state[V*H*64*64];
 *         uint16 out_softmax[T*H*64]; uint16 out_from_state[T*H*64]
 * Exit status 0 on success; otherwise the failing call and its detail on stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "spanla.h"

#define CHECK_CUDA(x)                                                                  \
  do {                                                                                 \
    cudaError_t e_ = (x);                                                              \
    if (e_ != cudaSuccess) {                                                           \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                         \
      return 2;                                                                        \
    }                                                                                  \
  } while (0)

#define CHECK_SPAN(x)                                                                  \
  do {                                                                                 \
    span_la_status s_ = (x);                                                           \
    if (s_ != SPAN_LA_OK) {                                                            \
      fprintf(stderr, "%s: %s (%s)\n", #x, span_la_status_string(s_),                  \
              span_la_last_error_detail());                                            \
      return 3;                                                                        \
    }                                                                                  \
  } while (0)

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s <input> <output>\n", argv[0]);
    return 1;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t hdr[4];
  if (!read_all(in, hdr, sizeof(hdr))) return 1;
  const int32_t T = hdr[0], H = hdr[1], V = hdr[2], B = hdr[3];
  int32_t* vcu = (int32_t*)malloc(sizeof(int32_t) * (V + 1));
  int32_t* bcu = (int32_t*)malloc(sizeof(int32_t) * (B + 1));
  int32_t* par = (int32_t*)malloc(sizeof(int32_t) * (B > 0 ? B : 1));
  const size_t n = (size_t)T * H * 64;
  uint16_t* host = (uint16_t*)malloc(3 * n * sizeof(uint16_t));
  if (!read_all(in, vcu, sizeof(int32_t) * (V + 1)) || !read_all(in, bcu, sizeof(int32_t) * (B + 1)) ||
      !read_all(in, par, sizeof(int32_t) * B) || !read_all(in, host, 3 * n * sizeof(uint16_t)))
    return 1;
  fclose(in);

  void *q, *k, *v, *out, *out_sm, *out_fs;
  float* state;
  CHECK_CUDA(cudaMalloc(&q, n * 2));
  CHECK_CUDA(cudaMalloc(&k, n * 2));
  CHECK_CUDA(cudaMalloc(&v, n * 2));
  CHECK_CUDA(cudaMalloc(&out, n * 2));
  CHECK_CUDA(cudaMalloc(&out_sm, n * 2));
  CHECK_CUDA(cudaMalloc(&out_fs, n * 2));
  CHECK_CUDA(cudaMalloc((void**)&state, (size_t)(V > 0 ? V : 1) * H * 4096 * sizeof(float)));
  CHECK_CUDA(cudaMemcpy(q, host, n * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k, host + n, n * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v, host + 2 * n, n * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(out, 0, n * 2));
  CHECK_CUDA(cudaMemset(out_sm, 0, n * 2));
  CHECK_CUDA(cudaMemset(out_fs, 0, n * 2));

  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));
  span_la_dims dims;
  dims.total_rows = T;
  dims.num_heads = H;
  dims.head_dim = 64;
  dims.dtype = SPAN_LA_BF16;
  CHECK_SPAN(span_la_pass(q, k, v, dims, vcu, V, bcu, B, par, out, state, stream));
  CHECK_SPAN(span_la_softmax_pass(q, k, v, dims, vcu, V, bcu, B, par, 0.0f, out_sm, NULL, stream));
  /* the branches again, from the view states the pass wrote (shards of a long request) */
  CHECK_SPAN(span_la_branches_from_state(state, V, q, k, v, dims, bcu, B, par, out_fs, stream));
  CHECK_SPAN(span_la_check(stream));

  uint16_t* res = (uint16_t*)malloc(n * 2);
  float* st = (float*)malloc((size_t)(V > 0 ? V : 1) * H * 4096 * sizeof(float));
  FILE* o = fopen(argv[2], "wb");
  if (!o) return 1;
  CHECK_CUDA(cudaMemcpy(res, out, n * 2, cudaMemcpyDeviceToHost));
  fwrite(res, 2, n, o);
  CHECK_CUDA(cudaMemcpy(st, state, (size_t)V * H * 4096 * sizeof(float), cudaMemcpyDeviceToHost));
  fwrite(st, sizeof(float), (size_t)V * H * 4096, o);
  CHECK_CUDA(cudaMemcpy(res, out_sm, n * 2, cudaMemcpyDeviceToHost));
  fwrite(res, 2, n, o);
  CHECK_CUDA(cudaMemcpy(res, out_fs, n * 2, cudaMemcpyDeviceToHost));
  fwrite(res, 2, n, o);
  fclose(o);
  printf("spanla_client: T=%d H=%d V=%d B=%d ok (library version %d)\n", T, H, V, B, span_la_version());
  return 0;
}
