// santa_tile.cuh -- row geometry of the K/V cache for the TMA-streaming kernels,
// and the V-row gather shared by the samplers.
#pragma once

#include "santa_common.cuh"

namespace santa {

// A row of D elements of type T, cut into 128-byte column boxes for TMA.
template <typename T, int D>
struct TileGeom {
    static constexpr int kES = int(sizeof(T));
    static constexpr int kRowBytes = D * kES;        // 128, 256 or 512
    static constexpr int kBoxes = kRowBytes / 128;   // 128-byte column boxes per row
    static constexpr int kBoxElems = 128 / kES;      // elements per box row
    static constexpr int kEV = 16 / kES;             // elements per 16-byte vector
    static constexpr int kPairs = kEV / 2;           // float pairs per 16-byte vector
    static constexpr int kNJ = D / kEV;              // 16-byte vectors per row
};

// Gather-average helper: adds V rows J (one per lane of `j`, the first n lanes)
// of one KV head to the lane's slice accumulator, up to 16 loads in flight.
template <typename T, int D>
__device__ __forceinline__ void gather_rows(float (&acc)[D / 32], const T *vrow0, size_t row_stride, int j, int n,
                                            int lane) {
    constexpr int kE = D / 32;
    for (int r0 = 0; r0 < n; r0 += 16) {
        RowSlice<T, D> rows[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int jr = __shfl_sync(kFull, j, (r0 + r) & 31);
            if (r0 + r < n) rows[r].load(vrow0 + size_t(jr) * row_stride, lane);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r0 + r < n) {
#pragma unroll
                for (int e = 0; e < kE; ++e) acc[e] += rows[r].v[e];
            }
    }
}

}  // namespace santa
