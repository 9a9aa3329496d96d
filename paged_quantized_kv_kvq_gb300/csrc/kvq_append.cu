// kvq_append.cu -- quantize-and-scatter of new tokens, per-channel
// calibration, and a canonical read-back of slots (sm_103a).
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990): each decode step appends the new token's K/V to
// the cache (§1.1) into fixed-size physical blocks (§2.2); K/V are stored with
// absmax-symmetric INT8 (per-token, per-channel or per-group-of-128/64 scales)
// or FP8 (§2.3, §3.3; e5m2 without a scale, the fp8_e5m2 KV dtype of
// xpshop.cn article-312 §三), or INT4 per group (§2.3 names it beside INT8 and
// FP8).  Scale = absmax/127 (INT8), absmax/7 (INT4) or absmax/448 (e4m3) in
// fp32 with an IEEE division; code = clamp(round_half_even(x / scale), +-127)
// (+-7 for INT4), or e4m3 round-to-nearest-even with saturation; an all-zero
// group stores scale 0 and zero codes.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kvq_common.cuh"
#include "kvq_context.h"
#include "kvq_internal.h"

namespace kvq {

constexpr int kAppendThreads = 128;

struct AppendParams {
  PoolView pool;
  const __half* k;
  const __half* v;
  const int64_t* slots;  // null: decode-step form, the slot comes from table/lens
  int64_t T;
  // decode-step form: token t is sequence t's new token, at position lens[t]-1
  const int* table;
  const int* lens;
  int max_blocks, max_ctx;
  int64_t x_stride;  // elements between consecutive tokens of k and v
};

__device__ __forceinline__ float absmax8(const __half2 (&x)[4]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a = fmaxf(a, fabsf(__low2float(x[i])));
    a = fmaxf(a, fabsf(__high2float(x[i])));
  }
  return a;
}

// INT8 code, returned biased (c + 128) as stored in the pool.
__device__ __forceinline__ uint8_t quant_i8(float x, float s) {
  if (s == 0.f) return static_cast<uint8_t>(kInt8Bias);
  float q = rintf(__fdiv_rn(x, s));
  q = fminf(fmaxf(q, -127.f), 127.f);
  return static_cast<uint8_t>(static_cast<int>(q) + 128);
}

// INT4 code, returned biased (c + 8) as stored in the pool.
__device__ __forceinline__ uint32_t quant_i4(float x, float s) {
  if (s == 0.f) return kInt4Bias;
  float q = rintf(__fdiv_rn(x, s));
  q = fminf(fmaxf(q, -7.f), 7.f);
  return static_cast<uint32_t>(static_cast<int>(q) + 8);
}

// Replace the nibbles under `mask` of a shared 32-bit word: other tokens own
// the word's other nibbles and may be written by other CTAs at the same time.
__device__ __forceinline__ void store_nibbles(char* word, uint32_t mask, uint32_t val) {
  uint32_t* w = reinterpret_cast<uint32_t*>(word);
  atomicAnd(w, ~mask);
  atomicOr(w, val);
}

__device__ __forceinline__ uint8_t quant_e4m3(float x, float s) {
  if (s == 0.f) return 0;
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3));
}

// One CTA per (token, K|V).  Each thread owns 8 consecutive channels of one
// kv head per iteration (a 16-byte load).
template <int FMT>
__global__ void __launch_bounds__(kAppendThreads) kvq_append_kernel(const AppendParams p) {
  const PoolView& pool = p.pool;
  const int64_t t = blockIdx.x;
  const int kv = blockIdx.y;
  // Launched as a programmatic dependent (decode step), wait for the previous
  // kernel's completion before reading anything; otherwise returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Only then may the dependent decode launch: everything before this append
  // on the stream has completed by now, so the decode may read context
  // lengths, the block table and every page this append does not write (all
  // but each sequence's last page) before its own griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The row's first 16-byte chunk of each thread is loaded alongside the slot
  // lookup (every token has its row, padding included), so the two round
  // trips overlap.
  const __half* x = (kv == 0 ? p.k : p.v) + t * p.x_stride;
  const int per = pool.Hkv * pool.D;
  const uint4 raw0 = threadIdx.x * 8 < per ? *reinterpret_cast<const uint4*>(x + threadIdx.x * 8)
                                           : make_uint4(0, 0, 0, 0);
  int64_t slot;
  if (p.slots != nullptr) {
    slot = p.slots[t];
  } else {
    // a length beyond max_ctx is flagged by the decode; nothing is written
    const int L = p.lens[t];
    if (L <= 0 || L > p.max_ctx) return;
    const int blk = p.table[t * p.max_blocks + (L - 1) / pool.bs];
    slot = blk < 0 ? pool.num_blocks * pool.bs : (int64_t)blk * pool.bs + (L - 1) % pool.bs;
  }
  if (slot < 0) return;
  if (slot >= pool.num_blocks * pool.bs) {
    if (threadIdx.x == 0) set_error(pool.err, ERR_RANGE);
    return;
  }
  const int64_t blk = slot / pool.bs;
  const int off = static_cast<int>(slot % pool.bs);
  const int sub = off >> 4, tt = off & 15;
  const int D = pool.D, Hkv = pool.Hkv;

  __shared__ float red[kAppendThreads / 32];
  float tok_scale = 0.f;
  if constexpr (FMT == FMT_INT8_TOKEN || FMT == FMT_FP8_TOKEN) {
    float a = 0.f;
    for (int c = threadIdx.x * 8; c < per; c += kAppendThreads * 8) {
      uint4 raw = c < kAppendThreads * 8 ? raw0 : *reinterpret_cast<const uint4*>(x + c);
      a = fmaxf(a, absmax8(*reinterpret_cast<__half2(*)[4]>(&raw)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int w = 1; w < kAppendThreads / 32; ++w) a = fmaxf(a, red[w]);
    tok_scale = a == 0.f ? 0.f : __fdiv_rn(a, FMT == FMT_FP8_TOKEN ? 448.f : 127.f);
    if (threadIdx.x == 0) pool.tok_scales[(blk * 2 + kv) * pool.bs + off] = tok_scale;
  }

  // Whole warps iterate together (the per-group reduction shuffles across
  // lanes); lanes past the end carry zeros and store nothing.
  for (int base = 0; base < per; base += kAppendThreads * 8) {
    const int c = base + threadIdx.x * 8;
    const bool act = c < per;
    const int h = act ? c / D : 0, d0 = act ? c - h * D : 0;
    char* page = pool.pages + (blk * Hkv + h) * pool.page_bytes;
    char* tile = page + (kv == 0 ? 0 : pool.code_bytes) + sub * pool.sub_bytes;
    uint4 raw = base == 0 ? raw0 : act ? *reinterpret_cast<const uint4*>(x + c) : make_uint4(0, 0, 0, 0);
    const __half2(&xv)[4] = *reinterpret_cast<const __half2(*)[4]>(&raw);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __low2float(xv[i]);
      f[2 * i + 1] = __high2float(xv[i]);
    }

    if constexpr (FMT == FMT_INT4_GROUP) {
      // group = g contiguous channels of this head: g/8 consecutive lanes
      const int lanes = pool.group >> 3;
      float a = absmax8(xv);
      for (int o = lanes >> 1; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      const float s = a == 0.f ? 0.f : __fdiv_rn(a, 7.f);
      uint32_t u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = quant_i4(f[i], s);
      if (!act) continue;
      if ((d0 % pool.group) == 0) {
        float* sc = reinterpret_cast<float*>(page + 2 * pool.code_bytes) +
                    (kv * pool.bs + off) * pool.ng + d0 / pool.group;
        *sc = s;
      }
      if (kv == 0) {
        // channels d0..d0+3 and d0+4..d0+7: four nibbles of one word each
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {
          uint32_t val = 0, mask = 0;
          int o = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            int sh;
            o = k_nibble(tt, d0 + 4 * hw + i, sh);
            val |= u[4 * hw + i] << sh;
            mask |= 0xFu << sh;
          }
          store_nibbles(tile + o, mask, val);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          int sh;
          const int o = v_nibble(tt, d0 + i, sh);
          store_nibbles(tile + o, 0xFu << sh, u[i] << sh);
        }
      }
    } else if constexpr (FMT == FMT_FP16) {
      if (!act) continue;
      const uint16_t* hb = reinterpret_cast<const uint16_t*>(&raw);
      if (kv == 0) {
        // channels d0..d0+3 and d0+4..d0+7 are two 4-element words
        *reinterpret_cast<uint2*>(tile + k_tile_offset(tt, d0, D, 2)) = make_uint2(raw.x, raw.y);
        *reinterpret_cast<uint2*>(tile + k_tile_offset(tt, d0 + 4, D, 2)) = make_uint2(raw.z, raw.w);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint16_t*>(tile + v_code_offset(tt, d0 + i, D, 2, pool.bs)) = hb[i];
      }
    } else {
      uint8_t code[8];
      if constexpr (FMT == FMT_INT8_GROUP) {
        // group = g contiguous channels of this head: g/8 consecutive lanes
        const int lanes = pool.group >> 3;
        float a = absmax8(xv);
        for (int o = lanes >> 1; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = a == 0.f ? 0.f : __fdiv_rn(a, 127.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = quant_i8(f[i], s);
        if (act && (d0 % pool.group) == 0) {
          float* sc = reinterpret_cast<float*>(page + 2 * pool.code_bytes) +
                      (kv * pool.bs + off) * pool.ng + d0 / pool.group;
          *sc = s;
        }
      } else if constexpr (FMT == FMT_INT8_TOKEN) {
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = quant_i8(f[i], tok_scale);
      } else if constexpr (FMT == FMT_FP8_TOKEN) {
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = quant_e4m3(f[i], tok_scale);
      } else if constexpr (FMT == FMT_FP8_E5M2) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          code[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(f[i], __NV_SATFINITE, __NV_E5M2));
      } else {  // FMT_INT8_CHANNEL
        const float* cs = pool.chan_scales + ((int64_t)kv * Hkv + h) * D + d0;
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = quant_i8(f[i], cs[i]);
      }
      if (!act) continue;
      if (kv == 0) {
        const uint32_t w0 = code[0] | (code[1] << 8) | (code[2] << 16) | ((uint32_t)code[3] << 24);
        const uint32_t w1 = code[4] | (code[5] << 8) | (code[6] << 16) | ((uint32_t)code[7] << 24);
        *reinterpret_cast<uint32_t*>(tile + k_tile_offset(tt, d0, D, 1)) = w0;
        *reinterpret_cast<uint32_t*>(tile + k_tile_offset(tt, d0 + 4, D, 1)) = w1;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          tile[v_code_offset(tt, d0 + i, D, 1, pool.bs)] = static_cast<char>(code[i]);
      }
    }
  }
}

// Per-channel calibration, pass 1: absmax of |x| per (K|V, channel) over a
// chunk of tokens, merged with an integer max on the (non-negative) float bits.
__global__ void kvq_calib_absmax_kernel(PoolView pool, const __half* k, const __half* v,
                                        int64_t T, int64_t chunk) {
  const int C = pool.Hkv * pool.D;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int kv = blockIdx.y;
  if (c >= C) return;
  const __half* x = kv == 0 ? k : v;
  const int64_t t0 = blockIdx.z * chunk, t1 = min(T, t0 + chunk);
  float a = 0.f;
  for (int64_t t = t0; t < t1; ++t) a = fmaxf(a, fabsf(__half2float(x[t * C + c])));
  atomicMax(reinterpret_cast<unsigned int*>(pool.chan_scales) + kv * C + c, __float_as_uint(a));
}

// Pass 2: scale = absmax / 127 (fp32 IEEE division), in place.
__global__ void kvq_calib_finish_kernel(PoolView pool) {
  const int n = 2 * pool.Hkv * pool.D;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  pool.chan_scales[i] = __fdiv_rn(pool.chan_scales[i], 127.f);
}

// Canonical read-back: codes [n][2][Hkv][D], scales per format.
__global__ void kvq_read_slots_kernel(PoolView pool, const int64_t* slots, int64_t n,
                                      void* codes_out, float* scales_out) {
  const int64_t i = blockIdx.x;
  const int kv = blockIdx.y;
  const int64_t slot = slots[i];
  if (slot < 0 || slot >= pool.num_blocks * pool.bs) {
    if (threadIdx.x == 0) set_error(pool.err, ERR_RANGE);
    return;
  }
  const int64_t blk = slot / pool.bs;
  const int off = static_cast<int>(slot % pool.bs);
  const int sub = off >> 4, tt = off & 15;
  const int D = pool.D, per = pool.Hkv * D, es = pool.esize;
  for (int c = threadIdx.x; c < per; c += blockDim.x) {
    const int h = c / D, d = c - h * D;
    const char* page = pool.pages + (blk * pool.Hkv + h) * pool.page_bytes;
    const char* tile = page + (kv == 0 ? 0 : pool.code_bytes) + sub * pool.sub_bytes;
    const int64_t dst = (i * 2 + kv) * per + c;
    if (pool.fmt == FMT_INT4_GROUP) {  // biased nibble -> signed code
      int sh;
      const int o = kv == 0 ? k_nibble(tt, d, sh) : v_nibble(tt, d, sh);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + o);
      reinterpret_cast<int8_t*>(codes_out)[dst] =
          static_cast<int8_t>(static_cast<int>((w >> sh) & 0xFu) - static_cast<int>(kInt4Bias));
      continue;
    }
    const int o = kv == 0 ? k_tile_offset(tt, d, D, es) : v_code_offset(tt, d, D, es, pool.bs);
    if (es == 2)
      reinterpret_cast<uint16_t*>(codes_out)[dst] = *reinterpret_cast<const uint16_t*>(tile + o);
    else  // INT8 codes are stored biased; hand back the signed code
      reinterpret_cast<uint8_t*>(codes_out)[dst] =
          *reinterpret_cast<const uint8_t*>(tile + o) ^
          (pool.fmt == FMT_FP8_TOKEN || pool.fmt == FMT_FP8_E5M2 ? 0u : kInt8Bias);
  }
  if (scales_out == nullptr) return;
  if (pool.fmt == FMT_INT8_GROUP || pool.fmt == FMT_INT4_GROUP) {
    const int ns = pool.Hkv * pool.ng;
    for (int c = threadIdx.x; c < ns; c += blockDim.x) {
      const int h = c / pool.ng, gi = c - h * pool.ng;
      const char* page = pool.pages + (blk * pool.Hkv + h) * pool.page_bytes;
      const float* sc = reinterpret_cast<const float*>(page + 2 * pool.code_bytes);
      scales_out[(i * 2 + kv) * ns + c] = sc[(kv * pool.bs + off) * pool.ng + gi];
    }
  } else if (pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN) {
    if (threadIdx.x == 0) scales_out[i * 2 + kv] = pool.tok_scales[(blk * 2 + kv) * pool.bs + off];
  }
}

// Copy-on-write: block dst[i] becomes a copy of block src[i] -- every kv
// head's page (codes and group scales) and, per-token formats, the block's
// token scales.  One CTA per (pair, kv head), 16-byte vector copies.
__global__ void kvq_copy_blocks_kernel(PoolView pool, const int* src, const int* dst, int n) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int s = src[i], d = dst[i];
  if (s < 0 || d < 0 || (int64_t)s >= pool.num_blocks || (int64_t)d >= pool.num_blocks) {
    if (h == 0 && threadIdx.x == 0) set_error(pool.err, ERR_RANGE);
    return;
  }
  const uint4* from = reinterpret_cast<const uint4*>(pool.pages + ((int64_t)s * pool.Hkv + h) * pool.page_bytes);
  uint4* to = reinterpret_cast<uint4*>(pool.pages + ((int64_t)d * pool.Hkv + h) * pool.page_bytes);
  for (int k = threadIdx.x; k < pool.page_bytes / 16; k += blockDim.x) to[k] = from[k];
  if (h == 0 && (pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN))
    for (int k = threadIdx.x; k < 2 * pool.bs; k += blockDim.x)
      pool.tok_scales[(int64_t)d * 2 * pool.bs + k] = pool.tok_scales[(int64_t)s * 2 * pool.bs + k];
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_copy_blocks(const PoolView& pool, const int* src, const int* dst, int n,
                               cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  kvq_copy_blocks_kernel<<<dim3(static_cast<unsigned>(n), pool.Hkv), 128, 0, st>>>(pool, src, dst, n);
  return phase_mark(st, cudaGetLastError());
}

cudaError_t launch_append(const PoolView& pool, const __half* k, const __half* v,
                          const int64_t* slots, int64_t T, cudaStream_t st) {
  return launch_step_append(pool, k, v, slots, T, nullptr, nullptr, 0, 0, st, false, 0);
}

namespace {

template <int FMT>
cudaError_t launch_append_fmt(const AppendParams& p, dim3 grid, cudaStream_t st, bool dependent) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAppendThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return phase_mark(st, cudaLaunchKernelEx(&cfg, kvq_append_kernel<FMT>, p));
}

}  // namespace

cudaError_t launch_step_append(const PoolView& pool, const __half* k, const __half* v,
                               const int64_t* slots, int64_t T, const int* table, const int* lens,
                               int max_blocks, int max_ctx, cudaStream_t st, bool dependent,
                               int64_t x_stride) {
  if (T == 0) return cudaSuccess;
  AppendParams p{pool, k, v, slots, T, table, lens, max_blocks, max_ctx,
                 x_stride > 0 ? x_stride : (int64_t)pool.Hkv * pool.D};
  dim3 grid(static_cast<unsigned>(T), 2);
  switch (pool.fmt) {
    case FMT_FP16: return launch_append_fmt<FMT_FP16>(p, grid, st, dependent);
    case FMT_INT8_TOKEN: return launch_append_fmt<FMT_INT8_TOKEN>(p, grid, st, dependent);
    case FMT_INT8_CHANNEL: return launch_append_fmt<FMT_INT8_CHANNEL>(p, grid, st, dependent);
    case FMT_INT8_GROUP: return launch_append_fmt<FMT_INT8_GROUP>(p, grid, st, dependent);
    case FMT_FP8_TOKEN: return launch_append_fmt<FMT_FP8_TOKEN>(p, grid, st, dependent);
    case FMT_INT4_GROUP: return launch_append_fmt<FMT_INT4_GROUP>(p, grid, st, dependent);
    case FMT_FP8_E5M2: return launch_append_fmt<FMT_FP8_E5M2>(p, grid, st, dependent);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_calibrate(const PoolView& pool, const __half* k, const __half* v, int64_t T,
                             cudaStream_t st) {
  const int C = pool.Hkv * pool.D;
  cudaError_t e = cudaMemsetAsync(pool.chan_scales, 0, sizeof(float) * 2 * C, st);
  if (e != cudaSuccess) return e;
  const int64_t chunk = 256;
  const int64_t nz = (T + chunk - 1) / chunk;
  dim3 grid((C + 255) / 256, 2, static_cast<unsigned>(nz < 65535 ? nz : 65535));
  const int64_t ch = (T + grid.z - 1) / grid.z;
  kvq_calib_absmax_kernel<<<grid, 256, 0, st>>>(pool, k, v, T, ch);
  e = phase_mark(st, cudaGetLastError());
  if (e != cudaSuccess) return e;
  kvq_calib_finish_kernel<<<(2 * C + 255) / 256, 256, 0, st>>>(pool);
  return phase_mark(st, cudaGetLastError());
}

cudaError_t launch_read_slots(const PoolView& pool, const int64_t* slots, int64_t n,
                              void* codes_out, float* scales_out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(n), 2);
  kvq_read_slots_kernel<<<grid, 256, 0, st>>>(pool, slots, n, codes_out, scales_out);
  return phase_mark(st, cudaGetLastError());
}

}  // namespace kvq
