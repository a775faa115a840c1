// kda_tma.cuh -- tensor-map (TMA) copies of the raw q, k, v, g_raw tiles.
//
// A map describes one [T_total, H, 128] bf16 input as a 3-D tensor
// {128 channels, H heads, T_total tokens} and copies boxes of
// 72 channels x 1 head x 16 tokens.  A chunk's tile of one tensor is two
// boxes, channels [0, 72) and [64, 136) (channels 128-135 lie outside the
// tensor and arrive as zeros), each 16 rows of 144 bytes: the row pitch of
// 144 bytes puts 8 consecutive rows on 8 different 4-bank groups, so
// ldmatrix reads of 8 rows are conflict-free, and rows r and r + 8 differ by
// a whole number of 128-byte lines.  Rows past the end of the tensor arrive
// as zeros; rows past the end of a sequence inside the tensor hold the next
// sequence's tokens, which the chunk builder overwrites with its fill values
// before it reads the tile (kda_chunk.cuh).
// The x coordinates are 0 and 64 channels (0 and 128 bytes, multiples of 16);
// the shared-memory destinations are 128-byte aligned.
#pragma once

#include <cuda.h>

#include "kda_common.cuh"

namespace kda {

constexpr int RAW_ROW = 144;             // bytes per tile row (72 bf16)
constexpr int RAW_BOX = 16 * RAW_ROW;    // one box: 16 rows (2304 B)
constexpr int RAW_TILE = 2 * RAW_BOX;    // one tensor's tile (4608 B)

// byte offset of (row r, channel d) in a raw tile
__host__ __device__ constexpr int raw_off(int r, int d) {
  return (d >> 6) * RAW_BOX + r * RAW_ROW + (d & 63) * 2;
}

// The maps of the four raw inputs, a kernel parameter (__grid_constant__).
struct RawMaps {
  CUtensorMap q, k, v, g;
};

// One box (x = first channel, h = head, t = first token) into shared memory,
// completing `bytes` on the mbarrier.  Issuing thread only.
__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int x, int h, int t,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(h), "r"(t), "r"(smem_u32(bar))
      : "memory");
}

// A chunk's tile of one tensor: its two boxes.
__device__ __forceinline__ void tma_tile(uint8_t* tile, const CUtensorMap* map, int h, int t0,
                                         uint64_t* bar) {
  tma_box(tile, map, 0, h, t0, bar);
  tma_box(tile + RAW_BOX, map, 64, h, t0, bar);
}

// Host: the map of one [T_total, H, 128] bf16 tensor (T_total >= 1, < 2^31).
cudaError_t make_raw_map(CUtensorMap* map, const void* base, int64_t T_total, int H);
// Host: the maps of q, k, v and (unless gate_scalar) g_raw; all zero when
// T_total is 0 (nothing is copied then).
cudaError_t make_raw_maps(RawMaps* maps, const void* q, const void* k, const void* v,
                          const void* g, int64_t T_total, int H, bool gate_scalar);

}  // namespace kda
