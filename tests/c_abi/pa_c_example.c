/*
 * The library used from C alone: include/pa.h and the CUDA runtime, no Python.
 *
 * A parallel-sampling batch is built with the native block manager (one prompt
 * forked into samples, each sample appending its own tokens; appends into the
 * shared partial block produce copy-on-write pairs), then on the GPU: the block
 * copies, the cache writes of every token, decode and split decode. Inputs and
 * outputs go to a binary file (argv[1]) that the test reads back and checks
 * against the oracle.
 *
 * Layout of the file (little-endian): int32 S, H, G, D, B, num_blocks, width;
 * float scale; int32 num_tokens, num_pairs, prompt_tokens; int64 slots[num_tokens];
 * int64 pairs[num_pairs][2]; float key[num_tokens][G][D], value[...];
 * float k_cache and v_cache [nb][G][B][D] before the step; int32
 * context_lens[S]; int32 block_tables[S][width]; float q[S][H][D]; k_cache and
 * v_cache after the step; float out[S][H][D]; float out_split[S][H][D].
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pa.h"

#define CHECK_CUDA(x)                                                       \
  do {                                                                      \
    cudaError_t e_ = (x);                                                   \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      return 1;                                                             \
    }                                                                       \
  } while (0)
#define CHECK_PA(x)                                                         \
  do {                                                                      \
    pa_status s_ = (x);                                                     \
    if (s_ != PA_OK) {                                                      \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, pa_status_string(s_)); \
      return 1;                                                             \
    }                                                                       \
  } while (0)

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;
static float next_normalish(void) { /* sum of 4 uniforms, centred: a cheap bell shape */
  float acc = 0.f;
  for (int i = 0; i < 4; ++i) {
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    acc += (float)((rng_state >> 40) & 0xffffff) / 16777216.0f;
  }
  return (acc - 2.0f) * 1.7f;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <output file>\n", argv[0]);
    return 2;
  }
  enum { S = 6, H = 8, G = 2, D = 64, B = 16, NB = 64, PROMPT = 45, TAIL = 20, T = 32 };
  const float scale = 1.0f / 8.0f;

  /* block manager: prompt of 45 tokens, 6 samples, 0..TAIL own tokens each (plus the new one) */
  pa_bm* bm = pa_bm_create(NB, B, 1);
  if (!bm) return 1;
  int32_t prompt_tokens[PROMPT];
  for (int i = 0; i < PROMPT; ++i) prompt_tokens[i] = 1000 + i;
  int32_t cached = 0;
  CHECK_PA(pa_bm_add_sequence(bm, 0, prompt_tokens, PROMPT, &cached));
  for (int s = 1; s < S; ++s) CHECK_PA(pa_bm_fork(bm, 0, s));

  /* every token of the batch gets K/V: the prompt's, then each sample's appended ones */
  int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * (PROMPT + S * (TAIL + 1)));
  int64_t pairs[S * (TAIL + 1)][2];
  int ntok = 0, npairs = 0;
  {
    int32_t width0 = pa_bm_block_table(bm, 0, NULL, 0);
    int32_t* t0 = (int32_t*)malloc(sizeof(int32_t) * width0);
    pa_bm_block_table(bm, 0, t0, width0);
    for (int i = 0; i < PROMPT; ++i) slots[ntok++] = (int64_t)t0[i / B] * B + i % B;
    free(t0);
  }
  for (int s = 0; s < S; ++s) {
    const int own = (s * 7) % (TAIL + 1);
    for (int i = 0; i <= own; ++i) {
      int64_t slot, src, dst;
      CHECK_PA(pa_bm_append(bm, s, 2000 + 100 * s + i, &slot, &src, &dst));
      slots[ntok++] = slot;
      if (src >= 0) {
        pairs[npairs][0] = src;
        pairs[npairs][1] = dst;
        ++npairs;
      }
    }
  }
  int32_t ctx[S], width = 0;
  for (int s = 0; s < S; ++s) {
    ctx[s] = (int32_t)pa_bm_context_len(bm, s);
    const int32_t n = pa_bm_block_table(bm, s, NULL, 0);
    if (n > width) width = n;
  }
  int32_t* tables = (int32_t*)calloc((size_t)S * width, sizeof(int32_t));
  for (int s = 0; s < S; ++s) pa_bm_block_table(bm, s, tables + (size_t)s * width, width);

  /* host data: pool garbage, K/V of every token, q */
  const size_t pool_elems = (size_t)NB * G * B * D;
  float* hk = (float*)malloc(pool_elems * sizeof(float));
  float* hv = (float*)malloc(pool_elems * sizeof(float));
  for (size_t i = 0; i < pool_elems; ++i) {
    hk[i] = next_normalish();
    hv[i] = next_normalish();
  }
  float* key = (float*)malloc(sizeof(float) * ntok * G * D);
  float* val = (float*)malloc(sizeof(float) * ntok * G * D);
  for (int i = 0; i < ntok * G * D; ++i) {
    key[i] = next_normalish();
    val[i] = next_normalish();
  }
  float* q = (float*)malloc(sizeof(float) * S * H * D);
  for (int i = 0; i < S * H * D; ++i) q[i] = next_normalish();
  float* hk0 = (float*)malloc(pool_elems * sizeof(float));
  float* hv0 = (float*)malloc(pool_elems * sizeof(float));
  memcpy(hk0, hk, pool_elems * sizeof(float));
  memcpy(hv0, hv, pool_elems * sizeof(float));

  /* device copies */
  float *dk, *dv, *dkey, *dval, *dq, *dout, *dout2;
  int64_t *dslots, *dpairs;
  int32_t *dctx, *dtab;
  void* ws;
  const int prompt_slots = PROMPT;  /* the prompt's tokens are written before the samples' */
  CHECK_CUDA(cudaMalloc((void**)&dk, pool_elems * sizeof(float)));
  CHECK_CUDA(cudaMalloc((void**)&dv, pool_elems * sizeof(float)));
  CHECK_CUDA(cudaMalloc((void**)&dkey, sizeof(float) * ntok * G * D));
  CHECK_CUDA(cudaMalloc((void**)&dval, sizeof(float) * ntok * G * D));
  CHECK_CUDA(cudaMalloc((void**)&dq, sizeof(float) * S * H * D));
  CHECK_CUDA(cudaMalloc((void**)&dout, sizeof(float) * S * H * D));
  CHECK_CUDA(cudaMalloc((void**)&dout2, sizeof(float) * S * H * D));
  CHECK_CUDA(cudaMalloc((void**)&dslots, sizeof(int64_t) * ntok));
  CHECK_CUDA(cudaMalloc((void**)&dpairs, sizeof(int64_t) * 2 * (npairs > 0 ? npairs : 1)));
  CHECK_CUDA(cudaMalloc((void**)&dctx, sizeof(int32_t) * S));
  CHECK_CUDA(cudaMalloc((void**)&dtab, sizeof(int32_t) * S * width));
  int32_t max_ctx = 0;
  for (int s = 0; s < S; ++s) max_ctx = ctx[s] > max_ctx ? ctx[s] : max_ctx;
  const size_t ws_bytes = pa_decode_split_workspace_bytes(S, H, D, max_ctx, T);
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemcpy(dk, hk, pool_elems * sizeof(float), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dv, hv, pool_elems * sizeof(float), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dkey, key, sizeof(float) * ntok * G * D, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dval, val, sizeof(float) * ntok * G * D, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dq, q, sizeof(float) * S * H * D, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dslots, slots, sizeof(int64_t) * ntok, cudaMemcpyHostToDevice));
  if (npairs) CHECK_CUDA(cudaMemcpy(dpairs, pairs, sizeof(int64_t) * 2 * npairs, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dctx, ctx, sizeof(int32_t) * S, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dtab, tables, sizeof(int32_t) * S * width, cudaMemcpyHostToDevice));

  /* the step: prompt writes, copy-on-write copies, the samples' writes, then attention */
  cudaStream_t st;
  CHECK_CUDA(cudaStreamCreate(&st));
  CHECK_PA(pa_reshape_and_cache(dkey, dval, dk, dv, dslots, prompt_slots, G, D, B, PA_LAYOUT_HND, NB, PA_F32, st));
  void* kp[1] = {dk};
  void* vp[1] = {dv};
  if (npairs) CHECK_PA(pa_copy_blocks(kp, vp, 1, dpairs, npairs, G, D, B, NB, PA_F32, st));
  CHECK_PA(pa_reshape_and_cache(dkey + (size_t)prompt_slots * G * D, dval + (size_t)prompt_slots * G * D, dk, dv,
                                dslots + prompt_slots, ntok - prompt_slots, G, D, B, PA_LAYOUT_HND, NB, PA_F32, st));
  CHECK_PA(pa_decode(dout, dq, dk, dv, dtab, width, dctx, S, H, G, D, B, PA_LAYOUT_HND, NB, scale, PA_F32, PA_F32,
                     st));
  CHECK_PA(pa_decode_split(dout2, dq, dk, dv, dtab, width, dctx, S, H, G, D, B, PA_LAYOUT_HND, NB, scale, PA_F32,
                           PA_F32, max_ctx, T, ws, ws_bytes, st));
  uint32_t err_bits = 0;
  CHECK_PA(pa_get_error(&err_bits, st));

  /* results back, to the file */
  float* out = (float*)malloc(sizeof(float) * S * H * D);
  float* out2 = (float*)malloc(sizeof(float) * S * H * D);
  CHECK_CUDA(cudaMemcpy(hk, dk, pool_elems * sizeof(float), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hv, dv, pool_elems * sizeof(float), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(out, dout, sizeof(float) * S * H * D, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(out2, dout2, sizeof(float) * S * H * D, cudaMemcpyDeviceToHost));
  FILE* f = fopen(argv[1], "wb");
  if (!f) return 1;
  const int32_t hdr[7] = {S, H, G, D, B, NB, width};
  fwrite(hdr, sizeof hdr, 1, f);
  fwrite(&scale, sizeof scale, 1, f);
  const int32_t counts[3] = {ntok, npairs, prompt_slots};
  fwrite(counts, sizeof counts, 1, f);
  fwrite(slots, sizeof(int64_t), ntok, f);
  fwrite(pairs, sizeof(int64_t), 2 * (size_t)npairs, f);
  fwrite(key, sizeof(float), (size_t)ntok * G * D, f);
  fwrite(val, sizeof(float), (size_t)ntok * G * D, f);
  fwrite(hk0, sizeof(float), pool_elems, f);
  fwrite(hv0, sizeof(float), pool_elems, f);
  fwrite(ctx, sizeof(int32_t), S, f);
  fwrite(tables, sizeof(int32_t), (size_t)S * width, f);
  fwrite(q, sizeof(float), S * H * D, f);
  fwrite(hk, sizeof(float), pool_elems, f);
  fwrite(hv, sizeof(float), pool_elems, f);
  fwrite(out, sizeof(float), S * H * D, f);
  fwrite(out2, sizeof(float), S * H * D, f);
  fclose(f);
  printf("ok: %d sequences, %d tokens written, %d copy-on-write pairs, device error bits %u\n", S, ntok, npairs,
         err_bits);
  pa_bm_destroy(bm);
  return err_bits == 0 ? 0 : 1;
}
