// Staging of one chunk's rows of a [C][H][128] bf16 row tensor into shared memory for the
// two-CTA forward / state-pass kernels and the gradient kernel.
//
// A chunk's local rows [0, 64) are, in order, replay rows (t < t_own, gathered through the
// plan's replay list), the sequence's own rows (t_own <= t < t_end, consecutive compact rows)
// and zero rows past the sequence end.
#pragma once
#include <cuda.h>

#include "tc_primitives.cuh"
#include "tensor_map.h"

namespace harts {

// One tensor's map: {128 channels, H, C}, boxes of 64 channels x 64 rows.
struct RowMaps {
    CUtensorMap box64;
};

__device__ __forceinline__ void cp_async_arrive_on(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(tc::smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_one(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::smem_addr(bar)) : "memory");
}

// Stage local rows [0, 64) of one chunk: own rows t in [t_own, t_end) are the compact rows
// own0 + t; rows below zero_below read as zero; other rows come from tab[t] (-1: zero).
// dst0 / dst1: the 1024-aligned tiles of channels 0-63 / 64-127 ([64 rows][128 B] each).
// A chunk of own rows only comes as one 64-row TMA box per channel half; any other chunk is
// gathered row by row by every thread (several small boxes per chunk measured slower than
// the gather).  All NT threads call this; it completes one phase of `bar`.
template <int NT>
__device__ __forceinline__ void stage_chunk_rows(const void *src, const RowMaps &maps, const int *tab, int32_t h,
                                                 int H, int t_own, int t_end, int32_t own0, int zero_below,
                                                 uint8_t *dst0, uint8_t *dst1, uint64_t *bar, bool defer = false) {
    const int tid = threadIdx.x;
    if (t_own == 0 && t_end == 64 && zero_below == 0) {
        if (tid == 0) {
            tc::mbar_expect_tx(bar, 16384);
            tc::tma_load_3d(dst0, &maps.box64, 0, h, own0, bar);
            tc::tma_load_3d(dst1, &maps.box64, 64, h, own0, bar);
        }
        return;
    }
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    for (int e = tid; e < 64 * 16; e += NT) {
        const int t = e >> 4, pc = e & 15;
        const int64_t row = t < zero_below ? -1 : tab[t];
        uint8_t *dst = (pc < 8 ? dst0 : dst1) + t * 128 + (((pc & 7) ^ (t & 7)) << 4);
        tc::cp_async16(dst, row >= 0 ? s8 + ((row * H + h) * 256 + pc * 16) : s8, row >= 0 ? 16u : 0u);
    }
    cp_async_arrive_on(bar);
    if (defer) return;                // the caller syncs once and then arrives (gather_done)
    __syncthreads();
    if (tid == 0) mbar_arrive_one(bar);
}

// The same staging done by one warp alone (a load warp): a full own chunk as two 64-row TMA
// boxes issued by lane 0, any other chunk gathered by the warp's 32 lanes.  All 32 lanes call
// this; it completes one phase of `bar`.
__device__ __forceinline__ void stage_chunk_rows_warp(const void *src, const RowMaps &maps, const int *tab,
                                                      int32_t h, int H, int t_own, int t_end, int32_t own0,
                                                      int zero_below, uint8_t *dst0, uint8_t *dst1, uint64_t *bar) {
    const int lane = threadIdx.x & 31;
    if (t_own == 0 && t_end == 64 && zero_below == 0) {
        if (lane == 0) {
            tc::mbar_expect_tx(bar, 16384);
            tc::tma_load_3d(dst0, &maps.box64, 0, h, own0, bar);
            tc::tma_load_3d(dst1, &maps.box64, 64, h, own0, bar);
        }
        return;
    }
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    for (int e = lane; e < 64 * 16; e += 32) {
        const int t = e >> 4, pc = e & 15;
        const int64_t row = t < zero_below ? -1 : tab[t];
        uint8_t *dst = (pc < 8 ? dst0 : dst1) + t * 128 + (((pc & 7) ^ (t & 7)) << 4);
        tc::cp_async16(dst, row >= 0 ? s8 + ((row * H + h) * 256 + pc * 16) : s8, row >= 0 ? 16u : 0u);
    }
    cp_async_arrive_on(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive_one(bar);
}

// Whether stage_chunk_rows gathers (and, with defer, leaves the arrive to gather_done).
__device__ __forceinline__ bool chunk_gathers(int t_own, int t_end, int zero_below) {
    return !(t_own == 0 && t_end == 64 && zero_below == 0);
}

// Host: the 64-row map of one row tensor.
inline bool encode_row_maps(RowMaps *m, const void *base, int H, int64_t C) {
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(C)};
    const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(H) * 256};
    const cuuint32_t box[3] = {64, 1, 64};
    return encode_bf16(&m->box64, base, 3, dims, strides, box);
}

}  // namespace harts
