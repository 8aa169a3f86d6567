// GB300 (sm_103a) per-block and per-channel cast: BF16 -> FP8 E4M3 / FP4
// E2M1 codes with one scale per 128 x 128 block, or one scale per channel
// (column) over all rows.
//
// TileKernels lists per-block and per-channel FP8/FP4 casting beside the
// per-token cast (README "Features"; hysenlabs page "TileKernels, TileLang
// kernels for MoE routing and low-precision quantization", section "Seven
// kernel families, from MoE routing to Sinkhorn normalisation").  The pages
// give no block shape; this library uses square 128 x 128 blocks.  The
// scale and code steps are the per-token cast's (tk_device.cuh): amax
// floored at 1e-4, r = amax / fmt_max in IEEE fp32 (optionally rounded up
// to a power of two, optionally stored as a UE8M0 byte), codes =
// RNE(sat(x / s)).  include/tk_cast.h states the contract.
//
// Design (memory-bound, no tensor cores):
//  * Tiles of 128 rows x 128 channels of BF16 (32 KiB) move into a ring of
//    shared-memory stages with 2-D TMA tensor copies
//    (cp.async.bulk.tensor.2d ... mbarrier::complete_tx) issued by one
//    producer thread per CTA.  Rows past M and channels past K arrive as
//    zeros (the tensor map's out-of-bounds fill), which changes no amax.
//  * One persistent CTA per SM (the ring takes most of shared memory):
//    6 stages and 3 consumer groups of 8 warps; group k takes this CTA's
//    tiles k, k+3, ...  A warp owns 16 rows of a tile, a lane 8 channels of
//    one of the two rows a warp step covers (16-byte shared loads; the 32
//    lanes read 512 contiguous bytes, free of bank conflicts).
//  * Per-block cast: a tile is one block.  Each warp loads its 8 x 16 bytes
//    into registers and releases the stage at once, reduces its amax by
//    shuffles, and the group combines its 8 warp maxima in shared memory
//    behind a named barrier; every warp then casts from registers.
//  * Per-channel cast, two launches on a caller workspace that holds the
//    column maxima and one counter per 128-channel strip, all zero between
//    calls:
//      1. column amax: per tile, each group reduces the 128 column maxima of
//         its 128 rows in shared memory and folds them into the workspace
//         with atomicMax on the fp32 bit patterns (non-negative floats order
//         like their bit patterns; max is exact and order-independent, so
//         the result does not depend on timing).  Its tile loads ask L2 to
//         keep the input (evict_last) for the second read;
//      2. cast: the tile pipeline again; with each tile the producer also
//         copies the tile's 128 column maxima (512 bytes) into the stage, the
//         group turns them into 128 scales and reciprocals in shared memory,
//         and each lane divides its 8 channels by their own scales.  The
//         tiles of the first block row write the caller's scale vector.
//         Each tile then counts itself in its strip's counter; the tile that
//         completes the count (every copy of the strip's maxima has landed)
//         sets the strip's maxima and counter back to zero, so the next call
//         needs no clearing pass (a memset between the launches would cost
//         a serialised gap of several microseconds).
//    Launch 2 is a programmatic dependent: it waits (griddepcontrol.wait)
//    for launch 1 before touching memory.
//  * Every wait is bounded in time; on expiry the kernel records a fault
//    code (tk_get_device_fault), stops, lets its own copies land and
//    returns.  The groups agree on stopping through a barrier reduction, so
//    no warp is left waiting at a named barrier.

#include <cuda.h>            // CUtensorMap and its enums (types only)
#include <cudaTypedefs.h>    // PFN_cuTensorMapEncodeTiled
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "tk_cast.h"
#include "tk_device.cuh"
#include "tk_internal.h"

namespace {

using tk_internal::aligned;
using tk_internal::cuda_fail;

constexpr int kTileCols = TK_BLOCK;                 // channels per tile (256 B rows)
constexpr int kTileRows = TK_BLOCK;                 // rows per tile (the block height)
constexpr int kRowBytes = kTileCols * 2;
constexpr int kTileBytes = kTileRows * kRowBytes;  // 32 KiB
constexpr int kAmaxBytes = kTileCols * 4;           // per-channel: the tile's column maxima
constexpr int kStageBytes = kTileBytes + kAmaxBytes;
static_assert(kStageBytes % 128 == 0, "tensor copies need 128-byte aligned stages");
constexpr int kGroupWarps = 8;
constexpr int kGroups = 3;
constexpr int kStages = 6;
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kPrefetchTiles = 4;
constexpr int kCtasPerSm = 1;
constexpr int kWarpRows = kTileRows / kGroupWarps;    // 16
constexpr int kSteps = kWarpRows / 2;                 // 2 rows per warp step
static_assert(kStages % kGroups == 0, "each stage belongs to one group");
static_assert(kTileCols == 16 * 8, "16 lanes x 8 channels cover a tile row");

// Shared memory, from a 1024-byte aligned base: the ring (each stage a tile
// plus a slot for its column maxima), the full and empty mbarriers, an abort
// flag, and per group two buffers of 8 x 128 floats for the cross-warp
// reductions (the per-channel cast keeps 128 scales and reciprocals there).
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kFlagOffset = kBarOffset + 16 * kStages;
constexpr int kRedOffset = kFlagOffset + 16;
constexpr int kRedFloats = 2 * kGroupWarps * kTileCols;   // per group
constexpr int kSmemBytes = kRedOffset + kGroups * kRedFloats * 4 + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KiB opt-in");

// The kernels this file builds (one template instance each).
constexpr int kBlockCast = 0;     // 128 x 128 blocks -> codes + block scales
constexpr int kColumnAmax = 1;    // column maxima into the workspace
constexpr int kChannelCast = 2;   // codes with per-column scales

__device__ unsigned int g_tile_fault;   // read and cleared via tk_get_device_fault

struct TileParams {
  uint8_t* codes;            // row m at codes + m * ld_codes
  int64_t ld_codes;
  uint8_t* scales;           // block: 4-byte words, block row rb at rb * ld_scales
  int64_t ld_scales;         //   words; channel: a vector of K entries
  unsigned int* col_amax;    // channel: [k_pad] fp32 bit patterns
  unsigned int* strip_count; // channel: [n_cb] tiles of each strip cast so far
  int M, K;
  int n_cb;                  // tile (block) columns: ceil(K / 128)
  int n_rb;                  // tile (block) rows: ceil(M / 128)
  int n_tiles;
  int k_pad;                 // n_cb * 128
  int ue8m0;                 // 1: packed exponent bytes, 0: fp32 words
};

// ------------------------------------------------------------ primitives

// L2 eviction priority of a kernel's tile loads (a hint; no effect on values).
template <int OP>
__device__ __forceinline__ uint64_t load_policy() {
  uint64_t pol;
  if constexpr (OP == kColumnAmax)        // read again by the cast: keep it
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else if constexpr (OP == kChannelCast)  // second read, mostly from L2
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  else                                    // read once
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map,
                                            int c, int r, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(r), "r"(bar), "l"(pol)
      : "memory");
}

// L2 prefetch of one tile.  A hint: it changes no memory and orders nothing.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c, int r) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(r) : "memory");
}

// Barrier `id` over one consumer group (its 8 warps), returning whether
// any of them passed `pred`.  Also orders the group's shared-memory writes
// before it with the reads after it.
__device__ __forceinline__ bool group_any(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(kGroupWarps * 32)
      : "memory");
  return r != 0;
}

// Eight channels (one 16-byte chunk of a tile row) -> codes at dst: 8 bytes
// (E4M3) or 4 bytes (E2M1, element 0 in the low nibble).  Channels 2k and
// 2k+1 are divided with the scale pair s2[k] and reciprocal pair i2[k]
// (quotient2 operands).
template <int FMT, bool POW2>
__device__ __forceinline__ void cast8(uint8_t* dst, const uint4& raw,
                                      const uint64_t (&s2)[4], const uint64_t (&i2)[4]) {
  float q[8];
  quotient2<POW2>(raw.x, s2[0], i2[0], q[0], q[1]);
  quotient2<POW2>(raw.y, s2[1], i2[1], q[2], q[3]);
  quotient2<POW2>(raw.z, s2[2], i2[2], q[4], q[5]);
  quotient2<POW2>(raw.w, s2[3], i2[3], q[6], q[7]);
  // Streaming stores (st.global.cs): nothing reads the codes back here, so
  // they are the first lines L2 gives up (measured: 128 x 128 blocks 93.4%
  // -> 94.6% of the copy bandwidth, the per-channel cast 56.3% -> 57.3%).
  if constexpr (FMT == TK_FMT_E4M3) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(dst),
                 "r"(cvt_e4m3x4(q[0], q[1], q[2], q[3])),
                 "r"(cvt_e4m3x4(q[4], q[5], q[6], q[7])) : "memory");
  } else {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(dst), "r"(cvt_e2m1x8(q)) : "memory");
  }
}

template <int FMT>
__device__ __forceinline__ uint8_t* code_ptr(const TileParams& p, int row, int col) {
  return p.codes + (int64_t)row * p.ld_codes + (FMT == TK_FMT_E4M3 ? col : col / 2);
}

// ------------------------------------------------------------ producer

template <int OP>
__device__ void tile_produce(const CUtensorMap* map, const TileParams& p,
                             uint32_t ring, uint32_t full0, uint32_t empty0,
                             volatile int* abort_flag, int my_tiles) {
  // This grid may have been launched before the previous kernel in the
  // stream finished (programmatic dependent launch).  The L2 prefetch of the
  // first tiles is a hint and may run before the wait (L2 is where the
  // previous kernel's writes land); every copy and, through the copies,
  // every consumer access follows the wait.
  const int n_prefetch = my_tiles < kPrefetchTiles ? my_tiles : kPrefetchTiles;
  for (int i = 0; i < n_prefetch; ++i) {
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    const int rb = t / p.n_cb;
    tma_prefetch_2d(map, (t - rb * p.n_cb) * kTileCols, rb * kTileRows);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t pol = load_policy<OP>();
  int issued = 0;
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kStages;
    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
    if (i >= kStages && !mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
      if (!*abort_flag) atomicOr(&g_tile_fault, kFaultProducerWait);
      *abort_flag = 1;
      break;
    }
    if (*abort_flag) break;
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    const int rb = t / p.n_cb;
    const int cb = t - rb * p.n_cb;
    const uint32_t full = full0 + 8 * s;
    const uint32_t dst = ring + (uint32_t)(s * kStageBytes);
    // the whole box counts, zero fill included
    mbar_arrive_expect_tx(full, OP == kChannelCast ? kStageBytes : kTileBytes);
    tma_load_2d(dst, map, cb * kTileCols, rb * kTileRows, full, pol);
    if constexpr (OP == kChannelCast)   // the tile's 128 column maxima (k_pad covers them)
      bulk_load(dst + kTileBytes, p.col_amax + cb * kTileCols, kAmaxBytes, full);
    issued = i + 1;
  }
  // Let every copy this thread issued land before the CTA can exit.
  for (int i = issued - 1; i >= 0 && i >= issued - kStages; --i) {
    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
    if (!mbar_wait(full0 + 8 * (i % kStages), ph, nullptr)) {
      atomicOr(&g_tile_fault, kFaultDrain);
      break;
    }
  }
}

// ------------------------------------------------------------ the kernel

template <int FMT, bool POW2, int OP>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
tile_cast_kernel(const __grid_constant__ CUtensorMap map, const TileParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t full0 = base + kBarOffset;
  const uint32_t empty0 = full0 + 8 * kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kFlagOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kGroupWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int my_tiles = (p.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) tile_produce<OP>(&map, p, base, full0, empty0, abort_flag, my_tiles);
    return;
  }

  const int group = warp / kGroupWarps;
  const int gw = warp % kGroupWarps;
  const int half = lane >> 4;          // which of a step's two rows
  const int chunk = lane & 15;         // 8-channel chunk of the tile row
  float* red = reinterpret_cast<float*>(smem + kRedOffset) + group * kRedFloats;

  for (int i = group, n = 0; i < my_tiles; i += kGroups, ++n) {
    const int s = i % kStages;
    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
    bool ok = mbar_wait(full0 + 8 * s, ph, abort_flag);
    if (!ok) {
      if (!*abort_flag) atomicOr(&g_tile_fault, kFaultConsumerWait);
      *abort_flag = 1;
    }
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    const int rb = t / p.n_cb;
    const int cb = t - rb * p.n_cb;
    const int r0 = rb * kTileRows + gw * kWarpRows + half;   // this lane's first row
    const int col = cb * kTileCols + chunk * 8;               // this lane's first channel

    const uint32_t stage = base + (uint32_t)(s * kStageBytes);
    float* buf = red + (n & 1) * (kGroupWarps * kTileCols);
    unsigned int strip_done = 0;   // tiles of this strip counted before this one
    if constexpr (OP == kChannelCast) {
      // This tile's copy of the strip's maxima has landed: count it now and
      // look at the result after the cast (the atomic's latency overlaps it).
      if (ok && gw == 0 && lane == 0) strip_done = atomicAdd(&p.strip_count[cb], 1u);
      // 128 column scales for this tile, one thread per column, before the
      // tile's data is read (the stage is released after the reads below)
      const int c = gw * 32 + lane;
      if (ok && c < kTileCols) {
        const float amax = __uint_as_float(
            reinterpret_cast<const unsigned int*>(smem + (stage - base) + kTileBytes)[c]);
        const GroupScale g = group_scale<FMT, POW2>(amax);
        buf[c] = g.s;
        buf[kTileCols + c] = quotient2_inv<POW2>(g);
        const int k = cb * kTileCols + c;
        if (rb == 0 && k < p.K) {            // each channel's scale written once
          if (p.ue8m0)
            p.scales[k] = (uint8_t)g.e;
          else
            reinterpret_cast<float*>(p.scales)[k] = g.s;
        }
      }
      if (group_any(1 + group, !ok)) break;
    }
    uint4 v[kSteps];
    if (ok) {
      const uint32_t src = stage +
                           (uint32_t)((gw * kWarpRows + half) * kRowBytes + chunk * 16);
#pragma unroll
      for (int j = 0; j < kSteps; ++j) v[j] = lds16(src + (uint32_t)(2 * j * kRowBytes));
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);   // data now in registers
    }

    if constexpr (OP == kBlockCast) {
      float m = 0.0f;
      if (ok) {
        uint32_t mm = bmax_chunk(v[0]);
#pragma unroll
        for (int j = 1; j < kSteps; ++j) mm = bmax2(mm, bmax_chunk(v[j]));
        m = bmax_value(mm);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) buf[gw] = m;
      }
      if (group_any(1 + group, !ok)) break;
      float bmax = buf[0];
#pragma unroll
      for (int w = 1; w < kGroupWarps; ++w) bmax = fmaxf(bmax, buf[w]);
      const GroupScale g = group_scale<FMT, POW2>(bmax);
      const float gi = quotient2_inv<POW2>(g);
      uint64_t sv[4], iv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sv[k] = pack_f32x2(g.s, g.s);
        iv[k] = pack_f32x2(gi, gi);
      }
      if (col < p.K) {
#pragma unroll
        for (int j = 0; j < kSteps; ++j) {
          const int row = r0 + 2 * j;
          if (row < p.M) cast8<FMT, POW2>(code_ptr<FMT>(p, row, col), v[j], sv, iv);
        }
      }
      if (gw == 0 && lane == 0) {
        if (p.ue8m0) {
          uint8_t* srow = p.scales + (int64_t)rb * p.ld_scales * 4;
          srow[cb] = (uint8_t)g.e;
          if (cb == p.n_cb - 1)   // unused bytes of the last packed word
            for (int b = cb + 1; (b & 3) != 0; ++b) srow[b] = 0;
        } else {
          reinterpret_cast<float*>(p.scales)[(int64_t)rb * p.ld_scales + cb] = g.s;
        }
      }
    } else if constexpr (OP == kColumnAmax) {
      if (ok) {
        // per channel pair, the largest magnitude over this lane's rows and
        // then over the other half-warp's rows (same channels)
        uint32_t cw[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
        for (int j = 1; j < kSteps; ++j) {
          cw[0] = bmax2(cw[0], v[j].x);
          cw[1] = bmax2(cw[1], v[j].y);
          cw[2] = bmax2(cw[2], v[j].z);
          cw[3] = bmax2(cw[3], v[j].w);
        }
        float cm[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t o = bmax2(cw[k], __shfl_xor_sync(0xFFFFFFFFu, cw[k], 16));
          cm[2 * k] = __uint_as_float((o << 16) & 0x7FFFFFFFu);
          cm[2 * k + 1] = __uint_as_float(o & 0x7FFF0000u);
        }
        if (half == 0) {
          float4* d = reinterpret_cast<float4*>(buf + gw * kTileCols + chunk * 8);
          d[0] = make_float4(cm[0], cm[1], cm[2], cm[3]);
          d[1] = make_float4(cm[4], cm[5], cm[6], cm[7]);
        }
      }
      if (group_any(1 + group, !ok)) break;
      const int c = gw * 32 + lane;          // one thread per tile column
      if (c < kTileCols) {
        float m = buf[c];
#pragma unroll
        for (int w = 1; w < kGroupWarps; ++w) m = fmaxf(m, buf[w * kTileCols + c]);
        const int k = cb * kTileCols + c;
        if (k < p.K && m > 0.0f) atomicMax(&p.col_amax[k], __float_as_uint(m));
      }
    } else {   // kChannelCast
      if (col < p.K) {
        const float4* sp = reinterpret_cast<const float4*>(buf + chunk * 8);
        const float4* ip = reinterpret_cast<const float4*>(buf + kTileCols + chunk * 8);
        const float4 s0 = sp[0], s1 = sp[1], i0 = ip[0], i1 = ip[1];
        const uint64_t sv[4] = {pack_f32x2(s0.x, s0.y), pack_f32x2(s0.z, s0.w),
                                pack_f32x2(s1.x, s1.y), pack_f32x2(s1.z, s1.w)};
        const uint64_t iv[4] = {pack_f32x2(i0.x, i0.y), pack_f32x2(i0.z, i0.w),
                                pack_f32x2(i1.x, i1.y), pack_f32x2(i1.z, i1.w)};
#pragma unroll
        for (int j = 0; j < kSteps; ++j) {
          const int row = r0 + 2 * j;
          if (row < p.M) cast8<FMT, POW2>(code_ptr<FMT>(p, row, col), v[j], sv, iv);
        }
      }
      // The last tile of the strip to count itself clears the strip for the
      // next call: every tile of the strip has its copy of the maxima.
      if (gw == 0) {
        const unsigned int done = __shfl_sync(0xFFFFFFFFu, strip_done, 0);
        if (done == (unsigned int)(p.n_rb - 1)) {
          for (int c = lane; c < kTileCols; c += 32) p.col_amax[cb * kTileCols + c] = 0u;
          if (lane == 0) p.strip_count[cb] = 0u;
        }
      }
    }
  }
}

// ------------------------------------------- per-channel dequantization
// y = code value * its channel's scale (one IEEE fp32 multiply), BF16
// (nearest even) or fp32 out.  An elementwise kernel: thread t of block
// (bx, by) owns the 16-channel column chunk bx * kDequantThreads + t, loads
// its 16 scales once, and walks rows by*R, (by + gridDim.y)*R, ... R at a
// time (R code loads in flight per thread).  Codes decode with the exact
// hardware conversions; each row chunk leaves as 32 B (BF16) or 64 B
// (fp32).  (Per-block codes dequantize on the per-token pipeline instead:
// there one scale serves a whole 16-channel chunk.)

struct ChannelDequantParams {
  const uint8_t* codes;      // row m at codes + m * ld_codes
  int64_t ld_codes;
  const uint8_t* scales;     // K fp32 words or K UE8M0 bytes, 16-byte aligned
  uint8_t* y;                // row m at y + m * ld_y_bytes
  int64_t ld_y_bytes;
  int M;
  int cpr;                   // 16-channel chunks per row
  int ue8m0;
  int y_fp32;
};

constexpr int kDequantThreads = 32;
constexpr int kDequantRows = 2;         // rows per thread per step
constexpr int kDequantCtasPerSm = 64;   // blocks per SM the grid aims at

template <int FMT>
__global__ void __launch_bounds__(kDequantThreads)
channel_dequant_kernel(const ChannelDequantParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int c = (int)blockIdx.x * kDequantThreads + (int)threadIdx.x;
  if (c >= p.cpr) return;
  const int col = c * 16;
  const int64_t code_off = FMT == TK_FMT_E4M3 ? col : col / 2;
  float s[16];
  if (p.ue8m0) {
    const uint4 e = *reinterpret_cast<const uint4*>(p.scales + col);
    const uint32_t w[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t b = (w[k / 4] >> (8 * (k % 4))) & 0xFFu;
      s[k] = __uint_as_float(b ? b << 23 : 0x00400000u);   // 2^(b-127)
    }
  } else {
    const float4* f = reinterpret_cast<const float4*>(p.scales) + col / 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = f[i];
      s[4 * i] = q.x;
      s[4 * i + 1] = q.y;
      s[4 * i + 2] = q.z;
      s[4 * i + 3] = q.w;
    }
  }
  for (int r0 = (int)blockIdx.y * kDequantRows; r0 < p.M;
       r0 += (int)gridDim.y * kDequantRows) {
    uint4 raw[kDequantRows];
#pragma unroll
    for (int j = 0; j < kDequantRows; ++j) {
      if (r0 + j >= p.M) break;
      const uint8_t* at = p.codes + (int64_t)(r0 + j) * p.ld_codes + code_off;
      if constexpr (FMT == TK_FMT_E4M3) {
        raw[j] = *reinterpret_cast<const uint4*>(at);
      } else {
        const uint2 h = *reinterpret_cast<const uint2*>(at);
        raw[j] = make_uint4(h.x, h.y, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < kDequantRows; ++j) {
      const int row = r0 + j;
      if (row >= p.M) break;
      float v[16];
      if constexpr (FMT == TK_FMT_E4M3) {
        decode16_e4m3(raw[j], v);
      } else {
        decode16_e2m1(make_uint2(raw[j].x, raw[j].y), v);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], s[k]);
      store_scaled16(p.y + (int64_t)row * p.ld_y_bytes + (int64_t)col * (p.y_fp32 ? 4 : 2),
                     v, 1.0f, p.y_fp32 != 0);
    }
  }
}

// ------------------------------------------------------------ host side

using TileKernel = void (*)(CUtensorMap, TileParams);

template <int OP>
TileKernel pick_tile(int fmt, bool pow2) {
  if (fmt == TK_FMT_E4M3)
    return pow2 ? tile_cast_kernel<TK_FMT_E4M3, true, OP> : tile_cast_kernel<TK_FMT_E4M3, false, OP>;
  return pow2 ? tile_cast_kernel<TK_FMT_E2M1, true, OP> : tile_cast_kernel<TK_FMT_E2M1, false, OP>;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Tensor map of a BF16 matrix [M rows][ld_x] with K valid channels, in
// 128 x 128 boxes, zero fill outside the matrix.
tk_status make_map(CUtensorMap* map, const void* x, int64_t M, int64_t K, int64_t ld_x) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return tk_internal::fail_message("cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld_x * 2)};
  const cuuint32_t box[2] = {(cuuint32_t)kTileCols, (cuuint32_t)kTileRows};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x),
                              dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return tk_internal::fail_message("cuTensorMapEncodeTiled rejected the input matrix");
  return TK_OK;
}

cudaLaunchConfig_t dependent_launch(cudaLaunchAttribute* attr, unsigned grid, unsigned threads,
                                    size_t smem, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

tk_status launch_tile(TileKernel fn, const CUtensorMap& map, const TileParams& p, void* stream) {
  int sms = 0;
  cudaError_t err = tk_internal::prepare_kernel(reinterpret_cast<const void*>(fn), kSmemBytes, &sms);
  if (err != cudaSuccess) return cuda_fail(err);
  const int slots = sms * kCtasPerSm;
  const int grid = p.n_tiles < slots ? p.n_tiles : slots;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = dependent_launch(attr, (unsigned)grid, kThreads, kSmemBytes, stream);
  err = cudaLaunchKernelEx(&cfg, fn, map, p);
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? TK_OK : cuda_fail(err);
}

// Checks shared by both entry points.
tk_status check_tile_args(int64_t M, int64_t K, int64_t ld_x, int fmt, int mode,
                          int64_t ld_codes) {
  if (fmt != TK_FMT_E4M3 && fmt != TK_FMT_E2M1) return TK_ERR_INVALID_ARG;
  if (mode < TK_SCALE_FP32 || mode > TK_SCALE_UE8M0_PACKED) return TK_ERR_INVALID_ARG;
  if (M < 0 || K <= 0 || K % 16 != 0) return TK_ERR_INVALID_ARG;
  if (M > (int64_t(1) << 30) || K > (int64_t(1) << 28)) return TK_ERR_UNSUPPORTED;
  const int64_t code_bytes = fmt == TK_FMT_E4M3 ? K : K / 2;
  if (ld_x < K || ld_codes < code_bytes) return TK_ERR_INVALID_ARG;
  return TK_OK;
}

tk_status check_tile_pointers(const void* x, int64_t ld_x, const void* codes, int64_t ld_codes,
                              const void* scales) {
  if (x == nullptr || codes == nullptr || scales == nullptr) return TK_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ld_x * 2) % 16 != 0 || !aligned(codes, 16) || ld_codes % 16 != 0 ||
      !aligned(scales, 4))
    return TK_ERR_MISALIGNED;
  return TK_OK;
}

TileParams base_params(int64_t M, int64_t K, int mode, void* codes, int64_t ld_codes,
                       void* scales) {
  TileParams p = {};
  p.codes = static_cast<uint8_t*>(codes);
  p.ld_codes = ld_codes;
  p.scales = static_cast<uint8_t*>(scales);
  p.M = (int)M;
  p.K = (int)K;
  p.n_cb = (int)((K + kTileCols - 1) / kTileCols);
  p.n_rb = (int)((M + kTileRows - 1) / kTileRows);
  p.k_pad = p.n_cb * kTileCols;
  p.ue8m0 = mode == TK_SCALE_UE8M0_PACKED ? 1 : 0;
  return p;
}

// --------------------------------------------- allocation-free variant
//
// tk_per_channel_cast_noalloc runs tk_per_channel_cast on a workspace that
// lives in static device memory instead of one the caller provides.  Callers
// that cannot allocate device memory at the point of the call use it: a C
// host without a caching allocator (cudaMalloc/cudaFree synchronise the
// device), or a serving loop that forbids allocation after warm-up.  Its
// limit is the size of the array below: at most kNoAllocMaxChannels
// channels.

constexpr int64_t kNoAllocMaxChannels = 65536;
constexpr size_t kNoAllocScratchBytes =
    (size_t)(4 * kNoAllocMaxChannels + (4 * (kNoAllocMaxChannels / TK_BLOCK) + 15) / 16 * 16);

static __device__ __align__(256) unsigned char g_channel_scratch[kNoAllocScratchBytes];

// Per device: the scratch's address, found and cleared once.
struct ScratchTable {
  std::mutex mu;
  static constexpr int kMaxDev = 64;
  void* addr[kMaxDev] = {};
};
ScratchTable g_scratch;

// The current device's scratch: on the first call for a device, its address
// (cudaGetSymbolAddress) and one clearing memset, since the per-channel
// workspace must be zero-filled before its first use.  That memset is
// synchronous, so the first call on each device must not be made while a
// stream is being captured.
tk_status channel_scratch(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= ScratchTable::kMaxDev) return TK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch.mu);
  if (g_scratch.addr[dev] == nullptr) {
    void* addr = nullptr;
    err = cudaGetSymbolAddress(&addr, g_channel_scratch);
    if (err != cudaSuccess) return cuda_fail(err);
    if (addr == nullptr || !aligned(addr, 256)) return TK_ERR_CUDA;
    err = cudaMemset(addr, 0, kNoAllocScratchBytes);
    if (err != cudaSuccess) return cuda_fail(err);
    g_scratch.addr[dev] = addr;
  }
  *out = g_scratch.addr[dev];
  return TK_OK;
}

tk_status channel_dequant(const void* codes, int64_t ld_codes, const void* scales,
                          int64_t M, int64_t K, int fmt, int mode, void* y, int64_t ld_y,
                          int out_dtype, void* stream) {
  const int64_t out_size = out_dtype == TK_OUT_FP32 ? 4 : 2;
  ChannelDequantParams p = {};
  p.codes = static_cast<const uint8_t*>(codes);
  p.ld_codes = ld_codes;
  p.scales = static_cast<const uint8_t*>(scales);
  p.y = static_cast<uint8_t*>(y);
  p.ld_y_bytes = ld_y * out_size;
  p.M = (int)M;
  p.cpr = (int)(K / 16);
  p.ue8m0 = mode == TK_SCALE_UE8M0_PACKED ? 1 : 0;
  p.y_fp32 = out_dtype == TK_OUT_FP32 ? 1 : 0;
  void (*fn)(ChannelDequantParams) = fmt == TK_FMT_E4M3 ? channel_dequant_kernel<TK_FMT_E4M3>
                                                        : channel_dequant_kernel<TK_FMT_E2M1>;
  int sms = 0;
  cudaError_t err = tk_internal::prepare_kernel(reinterpret_cast<const void*>(fn), 0, &sms);
  if (err != cudaSuccess) return cuda_fail(err);
  // x: the row's column chunks; y: row strides, an equal number per block,
  // enough to fill every SM
  const int64_t gx = (p.cpr + kDequantThreads - 1) / kDequantThreads;
  const int64_t row_steps = (M + kDequantRows - 1) / kDequantRows;
  const int64_t target = ((int64_t)sms * kDequantCtasPerSm + gx - 1) / gx;
  const int64_t iters = (row_steps + target - 1) / target;
  int64_t gy = (row_steps + iters - 1) / iters;
  if (gy > 65535) gy = 65535;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = dependent_launch(attr, 1u, kDequantThreads, 0, stream);
  cfg.gridDim = dim3((unsigned)gx, (unsigned)gy);
  err = cudaLaunchKernelEx(&cfg, fn, p);
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? TK_OK : cuda_fail(err);
}

tk_status check_dequant_args(int64_t M, int64_t K, int fmt, int mode, int64_t ld_codes,
                             int64_t ld_y, int out_dtype) {
  if (fmt != TK_FMT_E4M3 && fmt != TK_FMT_E2M1) return TK_ERR_INVALID_ARG;
  if (mode < TK_SCALE_FP32 || mode > TK_SCALE_UE8M0_PACKED) return TK_ERR_INVALID_ARG;
  if (out_dtype != TK_OUT_BF16 && out_dtype != TK_OUT_FP32) return TK_ERR_INVALID_ARG;
  if (M < 0 || K <= 0 || K % 16 != 0) return TK_ERR_INVALID_ARG;
  if (M > (int64_t(1) << 30) || K > (int64_t(1) << 28)) return TK_ERR_UNSUPPORTED;
  const int64_t code_bytes = fmt == TK_FMT_E4M3 ? K : K / 2;
  if (ld_codes < code_bytes || ld_y < K) return TK_ERR_INVALID_ARG;
  return TK_OK;
}

tk_status check_dequant_pointers(const void* codes, int64_t ld_codes, const void* scales,
                                 uintptr_t scale_align, const void* y, int64_t ld_y,
                                 int out_dtype) {
  if (codes == nullptr || scales == nullptr || y == nullptr) return TK_ERR_INVALID_ARG;
  const int64_t out_size = out_dtype == TK_OUT_FP32 ? 4 : 2;
  if (!aligned(codes, 16) || ld_codes % 16 != 0 || !aligned(scales, scale_align) ||
      !aligned(y, 16) || (ld_y * out_size) % 16 != 0)
    return TK_ERR_MISALIGNED;
  return TK_OK;
}

}  // namespace

namespace tk_internal {

tk_status tile_fault(unsigned int* fault, int clear) {
  cudaError_t err = cudaMemcpyFromSymbol(fault, g_tile_fault, sizeof(unsigned int));
  if (err != cudaSuccess) return cuda_fail(err);
  if (clear) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbol(g_tile_fault, &zero, sizeof(unsigned int));
    if (err != cudaSuccess) return cuda_fail(err);
  }
  return TK_OK;
}

}  // namespace tk_internal

extern "C" {

size_t tk_per_channel_workspace_bytes(int64_t K) {
  if (K <= 0 || K > (int64_t(1) << 28)) return 0;
  const int64_t n_cb = (K + kTileCols - 1) / kTileCols;
  return (size_t)(4 * n_cb * kTileCols + (4 * n_cb + 15) / 16 * 16);
}

tk_status tk_per_block_cast(const void* x, int64_t M, int64_t K, int64_t ld_x, int fmt,
                            int mode, void* codes, int64_t ld_codes, void* scales,
                            int64_t ld_scales, void* stream) {
  tk_status st = check_tile_args(M, K, ld_x, fmt, mode, ld_codes);
  if (st != TK_OK) return st;
  const int64_t n_cb = (K + kTileCols - 1) / kTileCols;
  const int64_t words = mode == TK_SCALE_UE8M0_PACKED ? (n_cb + 3) / 4 : n_cb;
  if (ld_scales < words) return TK_ERR_INVALID_ARG;
  if (M == 0) return TK_OK;
  st = check_tile_pointers(x, ld_x, codes, ld_codes, scales);
  if (st != TK_OK) return st;
  const int64_t n_tiles = (M + kTileRows - 1) / kTileRows * n_cb;
  if (n_tiles > INT32_MAX) return TK_ERR_UNSUPPORTED;

  TileParams p = base_params(M, K, mode, codes, ld_codes, scales);
  p.ld_scales = ld_scales;
  p.n_tiles = (int)n_tiles;
  CUtensorMap map;
  st = make_map(&map, x, M, K, ld_x);
  if (st != TK_OK) return st;
  return launch_tile(pick_tile<kBlockCast>(fmt, mode != TK_SCALE_FP32), map, p, stream);
}

tk_status tk_per_channel_cast(const void* x, int64_t M, int64_t K, int64_t ld_x, int fmt,
                              int mode, void* codes, int64_t ld_codes, void* scales,
                              void* workspace, size_t workspace_bytes, void* stream) {
  tk_status st = check_tile_args(M, K, ld_x, fmt, mode, ld_codes);
  if (st != TK_OK) return st;
  if (workspace_bytes < tk_per_channel_workspace_bytes(K)) return TK_ERR_INVALID_ARG;
  if (M == 0) return TK_OK;
  st = check_tile_pointers(x, ld_x, codes, ld_codes, scales);
  if (st != TK_OK) return st;
  if (workspace == nullptr) return TK_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return TK_ERR_MISALIGNED;
  const int64_t n_tiles = (M + kTileRows - 1) / kTileRows * ((K + kTileCols - 1) / kTileCols);
  if (n_tiles > INT32_MAX) return TK_ERR_UNSUPPORTED;

  TileParams p = base_params(M, K, mode, codes, ld_codes, scales);
  p.n_tiles = (int)n_tiles;
  p.col_amax = static_cast<unsigned int*>(workspace);
  p.strip_count = p.col_amax + p.k_pad;
  CUtensorMap map;
  st = make_map(&map, x, M, K, ld_x);
  if (st != TK_OK) return st;
  const bool pow2 = mode != TK_SCALE_FP32;

  // 1. column amax (the maxima start at +0, the bit pattern 0)
  st = launch_tile(tile_cast_kernel<TK_FMT_E4M3, false, kColumnAmax>, map, p, stream);
  if (st != TK_OK) return st;
  // 2. cast (column scales computed per tile from the maxima)
  return launch_tile(pick_tile<kChannelCast>(fmt, pow2), map, p, stream);
}

tk_status tk_per_channel_cast_noalloc(const void* x, int64_t M, int64_t K, int64_t ld_x,
                                      int fmt, int mode, void* codes, int64_t ld_codes,
                                      void* scales, void* stream) {
  tk_status st = check_tile_args(M, K, ld_x, fmt, mode, ld_codes);
  if (st != TK_OK) return st;
  if (K > kNoAllocMaxChannels) return TK_ERR_UNSUPPORTED;
  if (tk_per_channel_workspace_bytes(K) > kNoAllocScratchBytes) return TK_ERR_UNSUPPORTED;
  if (M == 0) return TK_OK;
  st = check_tile_pointers(x, ld_x, codes, ld_codes, scales);
  if (st != TK_OK) return st;
  void* scratch = nullptr;
  st = channel_scratch(&scratch);
  if (st != TK_OK) return st;
  return tk_per_channel_cast(x, M, K, ld_x, fmt, mode, codes, ld_codes, scales, scratch,
                             kNoAllocScratchBytes, stream);
}

tk_status tk_per_block_dequant(const void* codes, int64_t ld_codes, const void* scales,
                               int64_t ld_scales, int64_t M, int64_t K, int fmt, int mode,
                               void* y, int64_t ld_y, int out_dtype, void* stream) {
  tk_status st = check_dequant_args(M, K, fmt, mode, ld_codes, ld_y, out_dtype);
  if (st != TK_OK) return st;
  const int64_t n_cb = (K + kTileCols - 1) / kTileCols;
  if (ld_scales < (mode == TK_SCALE_UE8M0_PACKED ? (n_cb + 3) / 4 : n_cb))
    return TK_ERR_INVALID_ARG;
  if (M == 0) return TK_OK;
  st = check_dequant_pointers(codes, ld_codes, scales, 4, y, ld_y, out_dtype);
  if (st != TK_OK) return st;
  return tk_internal::block_dequant(codes, ld_codes, scales, ld_scales, M, K, fmt, mode, y,
                                   ld_y, out_dtype, stream);
}

tk_status tk_per_channel_dequant(const void* codes, int64_t ld_codes, const void* scales,
                                 int64_t M, int64_t K, int fmt, int mode, void* y,
                                 int64_t ld_y, int out_dtype, void* stream) {
  tk_status st = check_dequant_args(M, K, fmt, mode, ld_codes, ld_y, out_dtype);
  if (st != TK_OK) return st;
  if (M == 0) return TK_OK;
  st = check_dequant_pointers(codes, ld_codes, scales, 16, y, ld_y, out_dtype);
  if (st != TK_OK) return st;
  return channel_dequant(codes, ld_codes, scales, M, K, fmt, mode, y, ld_y, out_dtype, stream);
}

}  // extern "C"
