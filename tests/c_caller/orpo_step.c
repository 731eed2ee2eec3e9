/* A plain C caller of the head's C ABI: no C++ and no PyTorch.  It reads one step's inputs from
 * raw files, runs forward, loss and backward on the default stream with cudaMalloc'd buffers, and
 * writes the outputs back as raw files.
 *
 *   orpo_step <dir> M V d n_pairs softcap lambda
 *   inputs : dir/h.bin (bf16 [M,d]), W.bin (bf16 [V,d]), targets.bin (int32 [M]),
 *            mask.bin (uint8 [M]), seq_id.bin (int32 [M])
 *   outputs: dir/logp.bin, lse.bin (fp32 [M]), out.bin (fp32 [5]), dh.bin (fp32 [M,d]),
 *            dW.bin (fp32 [V,d]), status.txt (the device status word)
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "orpo_head.h"

static int load(const char* dir, const char* name, void* dst, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return 1;
  const size_t n = fread(dst, 1, bytes, f);
  fclose(f);
  return n != bytes;
}

static int save(const char* dir, const char* name, const void* src, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t n = fwrite(src, 1, bytes, f);
  fclose(f);
  return n != bytes;
}

static void* dev_copy(const void* host, size_t bytes) {
  void* p = NULL;
  if (cudaMalloc(&p, bytes ? bytes : 1) != cudaSuccess) return NULL;
  if (host && cudaMemcpy(p, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return p;
}

#define CHECK(call)                                                                 \
  do {                                                                              \
    int rc_ = (call);                                                               \
    if (rc_ != 0) {                                                                 \
      fprintf(stderr, "%s failed: %d %s\n", #call, rc_, orpo_status_string(rc_)); \
      return 1;                                                                     \
    }                                                                               \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s dir M V d n_pairs softcap lambda\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int64_t M = atoll(argv[2]), V = atoll(argv[3]), d = atoll(argv[4]);
  const int32_t P = atoi(argv[5]);
  const float softcap = (float)atof(argv[6]), lambda = (float)atof(argv[7]);

  const size_t hb = (size_t)(M * d * 2), wb = (size_t)(V * d * 2);
  void* h = malloc(hb);
  void* W = malloc(wb);
  int32_t* targets = malloc((size_t)M * 4);
  uint8_t* mask = malloc((size_t)M);
  int32_t* seq_id = malloc((size_t)M * 4);
  if (!h || !W || !targets || !mask || !seq_id) return 3;
  if (load(dir, "h.bin", h, hb) || load(dir, "W.bin", W, wb) || load(dir, "targets.bin", targets, (size_t)M * 4) ||
      load(dir, "mask.bin", mask, (size_t)M) || load(dir, "seq_id.bin", seq_id, (size_t)M * 4)) {
    fprintf(stderr, "cannot read the inputs in %s\n", dir);
    return 3;
  }

  const size_t ws_bytes = orpo_head_workspace_bytes(M, V, d);
  void* d_h = dev_copy(h, hb);
  void* d_W = dev_copy(W, wb);
  int32_t* d_targets = dev_copy(targets, (size_t)M * 4);
  uint8_t* d_mask = dev_copy(mask, (size_t)M);
  int32_t* d_seq = dev_copy(seq_id, (size_t)M * 4);
  float* d_logp = dev_copy(NULL, (size_t)M * 4);
  float* d_lse = dev_copy(NULL, (size_t)M * 4);
  float* d_out = dev_copy(NULL, 5 * 4);
  float* d_ell = dev_copy(NULL, (size_t)P * 2 * 4);
  float* d_g = dev_copy(NULL, (size_t)M * 4);
  float* d_dh = dev_copy(NULL, (size_t)(M * d) * 4);
  float* d_dW = dev_copy(NULL, (size_t)(V * d) * 4);
  void* d_ws = dev_copy(NULL, ws_bytes);
  int32_t* d_status = dev_copy(NULL, 4);
  if (!d_h || !d_W || !d_targets || !d_mask || !d_seq || !d_logp || !d_lse || !d_out || !d_ell || !d_g || !d_dh ||
      !d_dW || !d_ws || !d_status) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 4;
  }
  if (cudaMemset(d_status, 0, 4) != cudaSuccess) return 4;

  CHECK(orpo_head_fwd(d_h, d_W, d_targets, d_mask, M, V, d, softcap, d_logp, d_lse, d_ws, ws_bytes, d_status, NULL));
  CHECK(orpo_loss(d_logp, d_seq, d_mask, M, P, lambda, d_out, d_ell, d_g, d_status, NULL));
  CHECK(orpo_head_bwd(d_h, d_W, d_targets, d_mask, d_lse, d_g, M, V, d, softcap, d_dh, d_dW, 0, d_ws, ws_bytes,
                      d_status, NULL));
  if (cudaDeviceSynchronize() != cudaSuccess) {
    fprintf(stderr, "device error\n");
    return 5;
  }

  int32_t status = 0;
  float out[5];
  float* logp = malloc((size_t)M * 4);
  float* lse = malloc((size_t)M * 4);
  float* dh = malloc((size_t)(M * d) * 4);
  float* dW = malloc((size_t)(V * d) * 4);
  if (!logp || !lse || !dh || !dW) return 3;
  if (cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(logp, d_logp, (size_t)M * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(lse, d_lse, (size_t)M * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dh, d_dh, (size_t)(M * d) * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dW, d_dW, (size_t)(V * d) * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 5;
  char text[64];
  snprintf(text, sizeof text, "%d\n", (int)status);
  if (save(dir, "status.txt", text, strlen(text)) || save(dir, "out.bin", out, sizeof out) ||
      save(dir, "logp.bin", logp, (size_t)M * 4) || save(dir, "lse.bin", lse, (size_t)M * 4) ||
      save(dir, "dh.bin", dh, (size_t)(M * d) * 4) || save(dir, "dW.bin", dW, (size_t)(V * d) * 4))
    return 6;
  printf("ok loss %.9g status %d\n", out[0], (int)status);
  return 0;
}
