// kvq_common.cuh -- device-side layout, error bits and PTX helpers shared by
// the append, decode and read-back kernels (sm_103a).
//
// Pool layout in HBM (one pool per layer).  The pages prescribe none; this one
// is chosen so that one (block, kv head) of K and V -- everything one decode
// thread block needs for a block -- is one contiguous run that a single bulk
// copy brings into shared memory, and so that each lane of a warp then reads
// exactly the bytes its tensor-core fragments need with 16-byte loads.
//
//   header      : 256 B, int32 error word at offset 0
//   (INT8 codes are stored biased by +128, see kInt8Bias; INT4 codes as
//    nibbles biased by +8, see the INT4 sub-tile layout below)
//   pages       : [num_blocks][kv_heads] pages of page_bytes each:
//                   K codes : block_size/16 sub-tiles of 16 tokens x D
//                             (block size 8: half a sub-tile, see below)
//                   V codes : block_size/16 sub-tiles
//                   K scales: [block_size][D/group] fp32   (per-group only)
//                   V scales: [block_size][D/group] fp32   (per-group only)
//   token scales: [num_blocks][2][block_size] fp32         (per-token only)
//   chan scales : [2][kv_heads][D] fp32                    (per-channel only)
//
// Inside a 16-token sub-tile the codes are stored "fragment-native": element
// (t, d) of K sits where lane ((t%8)*4 + (d%16)/4) finds it in its 32-bit word
// w = (t/8)*(D/16) + d/16, byte e = d%4; element (t, d) of V sits in lane
// ((d%8)*4 + (t%8)/2), word w = (d/16)*2 + (d/8)%2, byte e = t%2 + 2*((t/8)%2).
// Words are packed four (one-byte codes) or two (fp16) per 16-byte chunk, and
// chunk c of every lane lies at c*512 + lane*16, so a warp reads a sub-tile
// with conflict-free 16-byte shared-memory loads.  With that order a lane's
// K word is exactly the A fragment of mma.m16n8k16 for Q.K (rows = tokens,
// k = channels permuted within each 16-channel step) and its V word is the A
// fragment of V^T for P.V (rows = channels, k = tokens).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace kvq {

enum Fmt : int {
  FMT_FP16 = 0,
  FMT_INT8_TOKEN = 1,
  FMT_INT8_CHANNEL = 2,
  FMT_INT8_GROUP = 3,
  FMT_FP8_TOKEN = 4,
  FMT_INT4_GROUP = 5,
  FMT_FP8_E5M2 = 6,
};

enum ErrBits : int {
  ERR_RANGE = 1,    // slot / block id outside the pool, or L > max_context_len
  ERR_TIMEOUT = 2,  // a bounded mbarrier wait gave up
};

constexpr int kHeaderBytes = 256;
constexpr int kWaitTries = 4000;  // bound of a pipeline wait: tries of <= 1 ms each, ~4 s
constexpr int kMaxDevicesApi = 64;

__host__ __device__ constexpr int fmt_esize(int fmt) { return fmt == FMT_FP16 ? 2 : 1; }

// Byte offset of element (t, d) of a K sub-tile (t in [0,16)).
__host__ __device__ inline int k_tile_offset(int t, int d, int D, int esize) {
  const int lane = (t & 7) * 4 + ((d & 15) >> 2);
  const int w = (t >> 3) * (D >> 4) + (d >> 4);
  const int e = d & 3;
  const int wpc = 4 / esize;  // words per 16-byte chunk
  return (w / wpc) * 512 + lane * 16 + (w % wpc) * 4 * esize + e * esize;
}

// Byte offset of element (t, d) of a V sub-tile (t in [0,16)).
__host__ __device__ inline int v_tile_offset(int t, int d, int D, int esize) {
  (void)D;
  const int lane = (d & 7) * 4 + ((t & 7) >> 1);
  const int w = (d >> 4) * 2 + ((d >> 3) & 1);
  const int e = (t & 1) + 2 * ((t >> 3) & 1);
  const int wpc = 4 / esize;
  return (w / wpc) * 512 + lane * 16 + (w % wpc) * 4 * esize + e * esize;
}

// Block size 8: a page holds half a sub-tile.  Its K codes are the first half
// of the K layout above (tokens 0..7 are the rows g of every lane, the first
// half of each lane's words).  Its V codes use their own order, since a V word
// above mixes tokens t and t+8: element (t, d) of an 8-token page sits in lane
// ((d%8)*4 + t/2), word w = d/16, byte e = t%2 + 2*((d/8)%2), so that a lane's
// word holds channels 16w + g and 16w + g + 8 at tokens 2j, 2j+1 -- the half of
// the V^T A fragment that one page supplies; the next page of the sequence
// supplies the other half (tokens 8 + 2j, 8 + 2j + 1).
__host__ __device__ inline int v_half_offset(int t, int d, int D, int esize) {
  (void)D;
  const int lane = (d & 7) * 4 + (t >> 1);
  const int w = d >> 4;
  const int e = (t & 1) + 2 * ((d >> 3) & 1);
  const int wpc = 4 / esize;
  return (w / wpc) * 512 + lane * 16 + (w % wpc) * 4 * esize + e * esize;
}

// Byte offset of element (t, d) of the V codes of a sub-tile (block size 16
// or more) or of an 8-token page.
__host__ __device__ inline int v_code_offset(int t, int d, int D, int esize, int bs) {
  return bs == 8 ? v_half_offset(t, d, D, esize) : v_tile_offset(t, d, D, esize);
}

// INT4 sub-tiles hold one 32-bit word per lane per 16-channel step: K word kk
// of a lane carries channels 16kk + 4j .. +3 of tokens g and g+8 (lane =
// 4g + j), V word mt carries tokens 2j, 2j+1, 2j+8, 2j+9 of channels 16mt + g
// and 16mt + g + 8.  Element e of a word is the nibble at bit nib_shift(e),
// an order in which one mask-and-or yields the fp16 pairs (e0,e1), (e4,e5)
// and a second, on the word shifted by 4, (e2,e3), (e6,e7).  Words are packed
// four per 16-byte chunk, chunk c of every lane at c*512 + lane*16.
__host__ __device__ inline int nib_shift(int e) { return (e & 1) * 16 + (e >> 1) * 4; }
__host__ __device__ inline int int4_word_offset(int lane, int wi) {
  return (wi >> 2) * 512 + lane * 16 + (wi & 3) * 4;
}
// Byte offset of the word holding element (t, d) of a K sub-tile, and its shift.
__host__ __device__ inline int k_nibble(int t, int d, int& shift) {
  shift = nib_shift((t >> 3) * 4 + (d & 3));
  return int4_word_offset((t & 7) * 4 + ((d & 15) >> 2), d >> 4);
}
// Same for a V sub-tile.
__host__ __device__ inline int v_nibble(int t, int d, int& shift) {
  shift = nib_shift((t & 1) + 2 * ((t >> 3) & 1) + 4 * ((d >> 3) & 1));
  return int4_word_offset((d & 7) * 4 + ((t & 7) >> 1), d >> 4);
}
constexpr uint32_t kInt4Bias = 8u;

// Plain-old-data view of a pool that kernels receive by value.
struct PoolView {
  char* pages;
  float* tok_scales;   // per-token: [NB][2][bs]
  float* chan_scales;  // per-channel: [2][Hkv][D]
  int* err;
  int64_t num_blocks;
  int bs, Hkv, D, fmt, group, ng, esize;
  int sub_bytes;    // bytes of one 16-token sub-tile: 16 * D * esize (INT4: 8 * D)
  int code_bytes;   // bytes of K (or V) codes in one page = bs * sub_bytes / 16
                    // (block size 8: half a sub-tile)
  int page_bytes;   // 2*code_bytes + (per-group) 2*bs*ng*4
};

__device__ __forceinline__ void set_error(int* err, int bits) { atomicOr(err, bits); }

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// One bounded attempt; true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return done != 0;
}

// Non-blocking test: true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Polls of the spinning phase of a bounded wait (non-blocking tests, each
// well under a microsecond) before it falls back to suspending tries.
constexpr int kSpinPolls = 20000;

// Bounded wait for the phase with this parity: first spin on non-blocking
// tests (a suspended thread is not always resumed the moment the phase
// completes), then up to `tries` suspending tries of <= 1 ms each.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int tries) {
  for (int i = 0; i < kSpinPolls; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  for (int i = 0; i < tries; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bulk (TMA, non-tensor) copy global -> shared, completion counted in bytes on
// the mbarrier.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// D = A * B + D, m16n8k16, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// INT8 codes are stored biased, as the byte u = c + 128 (c ^ 0x80), so that
// the conversion below needs no XOR.
constexpr uint32_t kInt8Bias = 0x80u;

// Four biased int8 codes (bytes 0..3 of w) -> two fp16x2: lo = (c0, c1),
// hi = (c2, c3).  Exact: u is placed in the low mantissa bits of 1024.0
// (0x6400 | u == 1024 + u), then 1152 = 1024 + 128 is subtracted.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t u, uint32_t& lo, uint32_t& hi) {
  const uint32_t l = prmt(u, 0x64646464u, 0x4140u);
  const uint32_t h = prmt(u, 0x64646464u, 0x4342u);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 lf = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  __half2 hf = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<uint32_t*>(&lf);
  hi = *reinterpret_cast<uint32_t*>(&hf);
}

// Four e5m2 codes -> two fp16x2.  An e5m2 code is the top byte of the fp16
// with the same value, so each byte only moves up: (c0,c1), (c2,c3).
__device__ __forceinline__ void e5m2x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = prmt(w, 0u, 0x1404u);
  hi = prmt(w, 0u, 0x3424u);
}

// Four e4m3 codes -> two fp16x2 (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint16_t wl = static_cast<uint16_t>(w & 0xFFFFu);
  const uint16_t wh = static_cast<uint16_t>(w >> 16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(wl));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(wh));
}

// Eight biased INT4 codes (nibbles in the order of nib_shift) -> four fp16x2
// pairs (e0,e1), (e2,e3), (e4,e5), (e6,e7).  Exact: a low nibble u placed in
// the mantissa of 1024.0 gives 1024 + u, less 1032 = u - 8; a high nibble
// (16u) gives 1024 + 16u, times 1/16 less 72 = u - 8 in one rounding-free
// fused multiply-add.
__device__ __forceinline__ void i4x8_to_h2x4(uint32_t w, uint32_t& p01, uint32_t& p23,
                                             uint32_t& p45, uint32_t& p67) {
  const uint32_t lo = 0x000F000Fu, hi = 0x00F000F0u, magic = 0x64006400u;
  const uint32_t a = (w & lo) | magic, b = (w & hi) | magic;
  const uint32_t w8 = w >> 8;
  const uint32_t c = (w8 & lo) | magic, d = (w8 & hi) | magic;
  const __half2 sub = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 mul = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 add = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&a), sub);
  __half2 r1 = __hfma2(*reinterpret_cast<const __half2*>(&b), mul, add);
  __half2 r2 = __hsub2(*reinterpret_cast<const __half2*>(&c), sub);
  __half2 r3 = __hfma2(*reinterpret_cast<const __half2*>(&d), mul, add);
  p01 = *reinterpret_cast<uint32_t*>(&r0);
  p23 = *reinterpret_cast<uint32_t*>(&r1);
  p45 = *reinterpret_cast<uint32_t*>(&r2);
  p67 = *reinterpret_cast<uint32_t*>(&r3);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace kvq
