/* The layer forward driven from plain C through include/moe_gb300.h: no Python, no torch.
 *
 * Usage: c_abi_forward DIR.  DIR holds layer.txt ("T d N K d_r d_s"), the bf16 tensors
 * x, W_router, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down as raw little-endian files
 * (<name>.bin, row-major, the layouts the header states), for a softmax router with L1
 * renormalisation, alpha = K, a constant shared gain of 1, no capacity and the fp16
 * intermediate format.  The program packs the down projections (moe_pack_weights), sizes
 * and prepares a workspace, runs moe_layer_forward on a stream of its own, reads the status
 * word and writes y.bin (fp32 [T][d]) and topk_idx.bin (int32 [T][K]) into DIR.  The
 * caller allocates every buffer; the library allocates nothing.  Exit status 0 on success. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe_gb300.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s.bin", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes);
  const size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s.bin", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

/* A device copy of a host file (bf16 elements). */
static void* upload(const char* dir, const char* name, size_t elems) {
  void* host = read_file(dir, name, elems * 2);
  if (!host) return NULL;
  void* dev = NULL;
  if (cudaMalloc(&dev, elems * 2) != cudaSuccess ||
      cudaMemcpy(dev, host, elems * 2, cudaMemcpyHostToDevice) != cudaSuccess)
    dev = NULL;
  free(host);
  return dev;
}

/* The packed fp16 copy of a down projection (MOE_H_F16). */
static void* pack(const void* W, int64_t elems, cudaStream_t st) {
  size_t bytes = 0;
  void* packed = NULL;
  if (moe_packed_weights_size(elems, &bytes) != MOE_OK) return NULL;
  if (cudaMalloc(&packed, bytes) != cudaSuccess) return NULL;
  if (moe_pack_weights(W, elems, packed, bytes, st) != MOE_OK) return NULL;
  return packed;
}

#define CHECK(cond, what)                                   \
  do {                                                      \
    if (!(cond)) {                                          \
      fprintf(stderr, "c_abi_forward: %s failed\n", what);  \
      return 1;                                             \
    }                                                       \
  } while (0)

int main(int argc, char** argv) {
  CHECK(argc == 2, "usage: c_abi_forward DIR");
  const char* dir = argv[1];
  char path[1024];
  snprintf(path, sizeof path, "%s/layer.txt", dir);
  FILE* f = fopen(path, "r");
  CHECK(f != NULL, "layer.txt");
  long long T;
  int d, N, K, dr, ds;
  const int n = fscanf(f, "%lld %d %d %d %d %d", &T, &d, &N, &K, &dr, &ds);
  fclose(f);
  CHECK(n == 6 && ds > 0, "layer.txt contents");

  moe_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.T = T;
  cfg.d_model = d;
  cfg.N = N;
  cfg.K = K;
  cfg.d_expert = dr;
  cfg.d_shared = ds;
  cfg.dtype = MOE_BF16;
  cfg.score = MOE_SCORE_SOFTMAX;
  cfg.norm = MOE_NORM_L1_SELECTED;
  cfg.alpha = (float)K;
  cfg.shared_mode = MOE_SHARED_CONST;
  cfg.shared_gain = 1.0f;
  cfg.cap_policy = MOE_CAP_NONE;
  cfg.capacity_factor = 1.0;
  cfg.num_ranks = 1;
  cfg.rho = NULL;
  cfg.norm_p = 2.0f;
  cfg.h_format = MOE_H_F16;
  cfg.h_scale_log2 = 0;

  cudaStream_t st;
  CHECK(cudaStreamCreate(&st) == cudaSuccess, "cudaStreamCreate");
  const size_t Ne = (size_t)N;
  void* x = upload(dir, "x", (size_t)T * d);
  void* W_router = upload(dir, "W_router", Ne * d);
  void* W_gate = upload(dir, "W_gate", Ne * dr * d);
  void* W_up = upload(dir, "W_up", Ne * dr * d);
  void* W_down = upload(dir, "W_down", Ne * d * dr);
  void* Ws_gate = upload(dir, "Ws_gate", (size_t)ds * d);
  void* Ws_up = upload(dir, "Ws_up", (size_t)ds * d);
  void* Ws_down = upload(dir, "Ws_down", (size_t)d * ds);
  CHECK(x && W_router && W_gate && W_up && W_down && Ws_gate && Ws_up && Ws_down, "inputs");
  void* Wd_packed = pack(W_down, (int64_t)Ne * d * dr, st);
  void* Wsd_packed = pack(Ws_down, (int64_t)d * ds, st);
  CHECK(Wd_packed && Wsd_packed, "moe_pack_weights");

  moe_weights w;
  memset(&w, 0, sizeof w);
  w.W_router = W_router;
  w.W_gate = W_gate;
  w.W_up = W_up;
  w.W_down = Wd_packed;
  w.Ws_gate = Ws_gate;
  w.Ws_up = Ws_up;
  w.Ws_down = Wsd_packed;

  float* y = NULL;
  int32_t* topk_idx = NULL;
  CHECK(cudaMalloc((void**)&y, (size_t)T * d * sizeof(float)) == cudaSuccess, "cudaMalloc y");
  CHECK(cudaMalloc((void**)&topk_idx, (size_t)T * K * sizeof(int32_t)) == cudaSuccess,
        "cudaMalloc topk_idx");
  moe_outputs out;
  memset(&out, 0, sizeof out);
  out.y = y;
  out.topk_idx = topk_idx;

  size_t ws_bytes = 0;
  void* ws = NULL;
  CHECK(moe_workspace_size(&cfg, &ws_bytes) == MOE_OK, "moe_workspace_size");
  CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess, "cudaMalloc workspace");   /* 256-B aligned */
  CHECK(moe_workspace_init(ws, ws_bytes, st) == MOE_OK, "moe_workspace_init");
  const moe_status s = moe_layer_forward(&cfg, &w, x, &out, ws, ws_bytes, st);
  if (s != MOE_OK) fprintf(stderr, "moe_layer_forward: %s\n", moe_status_string(s));
  CHECK(s == MOE_OK, "moe_layer_forward");
  int32_t code = -100;
  CHECK(moe_read_status(ws, &code, st) == MOE_OK && code == MOE_OK, "device status");

  float* y_host = (float*)malloc((size_t)T * d * sizeof(float));
  int32_t* idx_host = (int32_t*)malloc((size_t)T * K * sizeof(int32_t));
  CHECK(y_host && idx_host, "host buffers");
  CHECK(cudaMemcpy(y_host, y, (size_t)T * d * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess,
        "copy y");
  CHECK(cudaMemcpy(idx_host, topk_idx, (size_t)T * K * sizeof(int32_t), cudaMemcpyDeviceToHost) ==
            cudaSuccess,
        "copy topk_idx");
  CHECK(write_file(dir, "y", y_host, (size_t)T * d * sizeof(float)) == 0, "write y");
  CHECK(write_file(dir, "topk_idx", idx_host, (size_t)T * K * sizeof(int32_t)) == 0,
        "write topk_idx");
  printf("c_abi_forward: %s, T=%lld d=%d N=%d K=%d\n", moe_version(), T, d, N, K);
  return 0;
}
