// Decode attention of the sub-block that runs beside the MoE in a
// shortcut-connected MoE layer (dragon.c, "Shortcut-connected MoE": the MoE
// is computed on sub-block-0's normed hidden state and added at the end of
// sub-block-1, "a designed overlap window"; §10: "thread the MoE against
// sub-block-1's attention").  On the GPU the two run on separate streams;
// this kernel is the attention core of sub-block-1.
//
// o[b, h] = softmax(q[b, h] . K[b, :, c]^T / sqrt(d)) V[b, :, c] for every
// sequence b (its own cache of S keys), query head h and its key/value head
// c = h / (n_heads / n_kv_heads); bf16 q, K, V and o, f32 arithmetic.
// Split over the sequence (flash-decoding): CTA (chunk, c, b) scores its 256
// keys for the g = n_heads / n_kv_heads query heads of c, and writes the
// chunk's running maximum m, sum l and unnormalised f32 output; a second
// kernel merges the chunks: o = sum_c e^(m_c - m) acc_c / sum_c e^(m_c - m) l_c.
#include "common.cuh"
#include "kernels.h"

namespace fp8moe {

namespace {

constexpr int kAttD = 128;        // head dimension
constexpr int kAttChunk = 256;    // keys per CTA
constexpr int kAttThreads = 128;  // threads per CTA
constexpr int kAttMaxG = 8;       // query heads per key/value head

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = u4_word(v, i);
    f[2 * i] = bf16_bits_to_float(w & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_float(w >> 16);
  }
}

template <int G>
__global__ void __launch_bounds__(kAttThreads) attn_chunk_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kc,
    const __nv_bfloat16 *__restrict__ vc, int64_t S, int nh, int nkv, float scale,
    float *__restrict__ part, int n_chunks) {
  __shared__ float qs[G][kAttD];
  // scores / weights of the chunk; reused afterwards for the four warps'
  // partial outputs, [4][G][128] floats, twice the scores' size
  __shared__ float ps[G][2 * kAttChunk];
  __shared__ float red[G][kAttThreads / 32];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int chunk = blockIdx.x, c = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int64_t j0 = (int64_t)chunk * kAttChunk;
  const int nk = (int)((S - j0) < kAttChunk ? (S - j0) : kAttChunk);
  // the G query heads of key/value head c, pre-scaled by 1/sqrt(d)
  for (int i = t; i < G * kAttD; i += kAttThreads) {
    const int h = i / kAttD, dd = i % kAttD;
    qs[h][dd] = __bfloat162float(q[(b * nh + (int64_t)c * G + h) * kAttD + dd]) * scale;
  }
  __syncthreads();
  // ---- scores: thread t takes keys t and t + 128 of the chunk
  float mx[G];
#pragma unroll
  for (int h = 0; h < G; ++h) mx[h] = -INFINITY;
#pragma unroll
  for (int r = 0; r < kAttChunk / kAttThreads; ++r) {
    const int jj = r * kAttThreads + t;
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.f;
    if (jj < nk) {
      const uint4 *kr = reinterpret_cast<const uint4 *>(kc + ((b * S + j0 + jj) * nkv + c) * kAttD);
#pragma unroll 8
      for (int v8 = 0; v8 < kAttD / 8; ++v8) {
        float kf[8];
        bf16x8_to_f32(__ldg(kr + v8), kf);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int i = 0; i < 8; ++i) s[h] = fmaf(qs[h][8 * v8 + i], kf[i], s[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      ps[h][jj] = jj < nk ? s[h] : -INFINITY;
      mx[h] = fmaxf(mx[h], jj < nk ? s[h] : -INFINITY);
    }
  }
  // ---- chunk maximum and the sum of e^(s - m)
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float m = warp_max(mx[h]);
    if (lane == 0) red[h][wid] = m;
  }
  __syncthreads();
  float m[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = red[h][0];
    for (int w = 1; w < kAttThreads / 32; ++w) m[h] = fmaxf(m[h], red[h][w]);
  }
  __syncthreads();
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) lsum[h] = 0.f;
#pragma unroll
  for (int r = 0; r < kAttChunk / kAttThreads; ++r) {
    const int jj = r * kAttThreads + t;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float p = jj < nk ? __expf(ps[h][jj] - m[h]) : 0.f;
      ps[h][jj] = p;
      lsum[h] += p;
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float l = warp_sum(lsum[h]);
    if (lane == 0) red[h][wid] = l;
  }
  __syncthreads();
  // ---- P.V: thread t takes columns 8 (t % 16) .. + 7 of keys t / 16,
  // t / 16 + 8, ..: one 16-byte load per key, 8 keys per 128 threads
  const int cg = t & 15, kl = t >> 4;
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = 0.f;
  const int64_t vstride = (int64_t)nkv * kAttD;
  const __nv_bfloat16 *vrow = vc + ((b * S + j0) * nkv + c) * kAttD + 8 * cg;
#pragma unroll 4
  for (int jj = kl; jj < nk; jj += 8) {
    float vf[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(vrow + jj * vstride)), vf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pj = ps[h][jj];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(pj, vf[i], acc[h][i]);
    }
  }
  // sum over the 8 key lanes: the two of a warp by a shuffle, then the four
  // warps through shared memory (the scores are no longer needed)
  float *accs = &ps[0][0];  // [4 warps][G][128] = G * 2 * kAttChunk floats
  static_assert((kAttThreads / 32) * kAttD == 2 * kAttChunk, "partials fit the score buffer");
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v = acc[h][i] + __shfl_xor_sync(0xffffffffu, acc[h][i], 16);
      if ((lane >> 4) == 0) accs[(wid * G + h) * kAttD + 8 * cg + i] = v;
    }
  __syncthreads();
  // partial layout [b][head][chunk][d + 2]: acc, then m and l
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float *pp = part + (((b * nh + (int64_t)c * G + h) * n_chunks) + chunk) * (kAttD + 2);
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kAttThreads / 32; ++w) a += accs[(w * G + h) * kAttD + t];
    pp[t] = a;
    if (t == 0) {
      float l = 0.f;
      for (int w = 0; w < kAttThreads / 32; ++w) l += red[h][w];
      pp[kAttD] = m[h];
      pp[kAttD + 1] = l;
    }
  }
}

__global__ void __launch_bounds__(kAttThreads) attn_merge_kernel(const float *__restrict__ part,
                                                                 int n_chunks, int nh,
                                                                 __nv_bfloat16 *__restrict__ o) {
  const int64_t bh = blockIdx.x;  // b * nh + h
  const int t = threadIdx.x;
  const float *pp = part + bh * n_chunks * (kAttD + 2);
  float m = -INFINITY;
  for (int ch = 0; ch < n_chunks; ++ch) m = fmaxf(m, pp[ch * (kAttD + 2) + kAttD]);
  float l = 0.f, acc = 0.f;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const float w = __expf(pp[ch * (kAttD + 2) + kAttD] - m);
    l = fmaf(w, pp[ch * (kAttD + 2) + kAttD + 1], l);
    acc = fmaf(w, pp[ch * (kAttD + 2) + t], acc);
  }
  o[bh * kAttD + t] = __float2bfloat16_rn(acc / l);
}

}  // namespace

int64_t attention_chunks(int64_t S) { return (S + kAttChunk - 1) / kAttChunk; }

cudaError_t launch_decode_attention(const __nv_bfloat16 *q, const __nv_bfloat16 *kc,
                                    const __nv_bfloat16 *vc, int64_t B, int64_t S, int nh, int nkv,
                                    int d, float *part, __nv_bfloat16 *o, cudaStream_t s) {
  if (d != kAttD || nkv <= 0 || nh % nkv != 0) return cudaErrorInvalidValue;
  const int g = nh / nkv;
  const int n_chunks = (int)attention_chunks(S);
  const dim3 grid((unsigned)n_chunks, (unsigned)nkv, (unsigned)B);
  const float scale = 1.0f / sqrtf((float)d);
  switch (g) {
    case 1: attn_chunk_kernel<1><<<grid, kAttThreads, 0, s>>>(q, kc, vc, S, nh, nkv, scale, part, n_chunks); break;
    case 2: attn_chunk_kernel<2><<<grid, kAttThreads, 0, s>>>(q, kc, vc, S, nh, nkv, scale, part, n_chunks); break;
    case 4: attn_chunk_kernel<4><<<grid, kAttThreads, 0, s>>>(q, kc, vc, S, nh, nkv, scale, part, n_chunks); break;
    case 8: attn_chunk_kernel<8><<<grid, kAttThreads, 0, s>>>(q, kc, vc, S, nh, nkv, scale, part, n_chunks); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_merge_kernel<<<(unsigned)(B * nh), kAttThreads, 0, s>>>(part, n_chunks, nh, o);
  return cudaGetLastError();
}

}  // namespace fp8moe
