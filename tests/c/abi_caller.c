/*
 * A plain C caller of liblrm: the whole recalibration path through the C ABI
 * on buffers from cudaMalloc, with no Python in the call path.
 *
 *   abi_caller --probe          create a context; prints the status (on a
 *                               machine without a GB300 the call fails cleanly)
 *   abi_caller <in> <out>       read a layer from <in>, run route stats, score,
 *                               select, compact, dgrad and wgrad on stream 0,
 *                               write the results to <out>
 *
 * <in>:  int32 T, E, k, h, I, cf_num, cf_den, rho_num, rho_den, max_rows (the
 *        caller's expectation; the program sizes its buffers with lrm_max_rows
 *        and fails if the two differ); then
 *        logits f32[T*E], expert_idx i32[T*k], alpha f32[T*k], g bf16[T*h],
 *        phi bf16[T*k*I], W bf16[E*h*I]
 * <out>: uint32 device status; f32 score[T*k]; int32 sel_offsets[E+1],
 *        sel_ids[max_rows]; bf16 dphi_c[max_rows*I]; f32 dW[E*h*I]; the route
 *        summary struct
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "lrm.h"

#define CHECK_LRM(call)                                                          \
  do {                                                                           \
    lrm_status s_ = (call);                                                      \
    if (s_ != LRM_OK) {                                                          \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #call, lrm_status_string(s_)); \
      return 2;                                                                  \
    }                                                                            \
  } while (0)
#define CHECK_CUDA(call)                                                         \
  do {                                                                           \
    cudaError_t e_ = (call);                                                     \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
      return 3;                                                                  \
    }                                                                            \
  } while (0)

static void* read_block(FILE* f, size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (p && bytes && fread(p, 1, bytes, f) != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc == 2 && strcmp(argv[1], "--probe") == 0) {
    lrm_ctx* ctx = NULL;
    lrm_status s = lrm_create(0, &ctx);
    printf("abi %d create %s\n", (int)lrm_abi_version(), lrm_status_string(s));
    if (s == LRM_OK) lrm_destroy(ctx);
    return 0;
  }
  if (argc != 3) {
    fprintf(stderr, "usage: %s --probe | <in> <out>\n", argv[0]);
    return 1;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t hdr[10];
  if (fread(hdr, sizeof(int32_t), 10, in) != 10) return 1;
  const lrm_dims dims = {hdr[0], hdr[1], hdr[2], hdr[3], hdr[4]};
  int32_t max_rows = 0;
  CHECK_LRM(lrm_max_rows(dims, hdr[5], hdr[6], hdr[7], hdr[8], &max_rows));
  if (max_rows != hdr[9]) {
    fprintf(stderr, "lrm_max_rows gave %d, the input expects %d\n", (int)max_rows, (int)hdr[9]);
    return 4;
  }
  const size_t T = (size_t)dims.T, E = (size_t)dims.E, k = (size_t)dims.k, h = (size_t)dims.h, I = (size_t)dims.I;
  const size_t N = T * k;
  void* h_logits = read_block(in, T * E * 4);
  void* h_idx = read_block(in, N * 4);
  void* h_alpha = read_block(in, N * 4);
  void* h_g = read_block(in, T * h * 2);
  void* h_phi = read_block(in, N * I * 2);
  void* h_W = read_block(in, E * h * I * 2);
  fclose(in);
  if (!h_logits || !h_idx || !h_alpha || !h_g || !h_phi || !h_W) return 1;

  lrm_ctx* ctx = NULL;
  CHECK_LRM(lrm_create(0, &ctx));
  float* logits = (float*)to_device(h_logits, T * E * 4);
  int32_t* idx = (int32_t*)to_device(h_idx, N * 4);
  float* alpha = (float*)to_device(h_alpha, N * 4);
  uint16_t* g = (uint16_t*)to_device(h_g, T * h * 2);
  uint16_t* phi = (uint16_t*)to_device(h_phi, N * I * 2);
  uint16_t* W = (uint16_t*)to_device(h_W, E * h * I * 2);
  if (!logits || !idx || !alpha || !g || !phi || !W) return 3;

  size_t ws_route = 0, ws_select = 0;
  CHECK_LRM(lrm_workspace_size(ctx, LRM_OP_ROUTE_STATS, dims, &ws_route));
  CHECK_LRM(lrm_workspace_size(ctx, LRM_OP_SELECT, dims, &ws_select));
  const size_t R = max_rows > 0 ? (size_t)max_rows : 1;
  int32_t *counts, *offsets, *bucket, *quota, *sel_offsets, *sel_ids;
  float *P, *f, *score, *alpha_c, *dW;
  uint16_t *delta_c, *phi_c, *dphi_c;
  lrm_route_summary* summary;
  void *wsr, *wss;
  CHECK_CUDA(cudaMalloc((void**)&counts, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&offsets, (E + 1) * 4));
  CHECK_CUDA(cudaMalloc((void**)&bucket, (N ? N : 1) * 4));
  CHECK_CUDA(cudaMalloc((void**)&quota, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&P, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&f, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&summary, sizeof(lrm_route_summary)));
  CHECK_CUDA(cudaMalloc(&wsr, ws_route ? ws_route : 256));
  CHECK_CUDA(cudaMalloc(&wss, ws_select ? ws_select : 256));
  CHECK_CUDA(cudaMalloc((void**)&score, (N ? N : 1) * 4));
  CHECK_CUDA(cudaMalloc((void**)&sel_offsets, (E + 1) * 4));
  CHECK_CUDA(cudaMalloc((void**)&sel_ids, R * 4));
  CHECK_CUDA(cudaMalloc((void**)&delta_c, R * h * 2));
  CHECK_CUDA(cudaMalloc((void**)&phi_c, R * I * 2));
  CHECK_CUDA(cudaMalloc((void**)&alpha_c, R * 4));
  CHECK_CUDA(cudaMalloc((void**)&dphi_c, R * I * 2));
  CHECK_CUDA(cudaMalloc((void**)&dW, E * h * I * 4));

  CHECK_LRM(lrm_route_stats(ctx, logits, idx, dims, hdr[5], hdr[6], hdr[7], hdr[8], counts, offsets, bucket, P, f,
                            quota, summary, wsr, ws_route, NULL));
  CHECK_LRM(lrm_score(ctx, g, phi, alpha, dims, score, NULL));
  CHECK_LRM(lrm_select(ctx, score, offsets, bucket, quota, dims, max_rows, sel_offsets, sel_ids, wss, ws_select, NULL));
  CHECK_LRM(lrm_compact(ctx, g, phi, alpha, sel_offsets, sel_ids, dims, max_rows, delta_c, phi_c, alpha_c, NULL));
  CHECK_LRM(lrm_grouped_dgrad(ctx, delta_c, W, sel_offsets, dims, max_rows, dphi_c, NULL));
  CHECK_LRM(lrm_grouped_wgrad(ctx, delta_c, phi_c, sel_offsets, dims, max_rows, 0, dW, NULL));
  uint32_t flags = 0;
  CHECK_LRM(lrm_get_device_status(ctx, NULL, &flags));

  float* o_score = (float*)malloc((N ? N : 1) * 4);
  int32_t* o_off = (int32_t*)malloc((E + 1) * 4);
  int32_t* o_ids = (int32_t*)malloc(R * 4);
  uint16_t* o_dphi = (uint16_t*)malloc(R * I * 2);
  float* o_dW = (float*)malloc(E * h * I * 4);
  lrm_route_summary o_sum;
  if (!o_score || !o_off || !o_ids || !o_dphi || !o_dW) return 1;
  CHECK_CUDA(cudaMemcpy(o_score, score, N * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(o_off, sel_offsets, (E + 1) * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(o_ids, sel_ids, R * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(o_dphi, dphi_c, R * I * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(o_dW, dW, E * h * I * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&o_sum, summary, sizeof o_sum, cudaMemcpyDeviceToHost));
  FILE* out = fopen(argv[2], "wb");
  if (!out) return 1;
  fwrite(&flags, 4, 1, out);
  fwrite(o_score, 4, N, out);
  fwrite(o_off, 4, E + 1, out);
  fwrite(o_ids, 4, R, out);
  fwrite(o_dphi, 2, R * I, out);
  fwrite(o_dW, 4, E * h * I, out);
  fwrite(&o_sum, sizeof o_sum, 1, out);
  fclose(out);
  CHECK_LRM(lrm_destroy(ctx));
  return 0;
}
