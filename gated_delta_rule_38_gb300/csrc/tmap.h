// Host-side creation of TMA tensor maps (driver entry point looked up through the runtime).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

// The tensor-map encoder is a driver call and needs a current context on the calling thread, which the
// runtime binds only lazily: a thread that has made no runtime call yet (a framework's worker thread) has
// none.  With no current context this makes the current device's primary context current (cudaSetDevice);
// a context the caller made current is left in place.
cudaError_t ensure_context();

// A rank-3 tiled map over a row-major [dim2][dim1][dim0] tensor of 16-bit elements (dim0 contiguous),
// strides in bytes for dims 1 and 2, a box of box0 x box1 x box2 elements, 128-byte swizzle, zero fill
// outside the tensor.  Returns false when the driver refuses the map.
bool make_tmap_3d(CUtensorMap *map, const void *base, bool bf16, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                  uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2);

// A token tensor [tokens][heads][cols] (16-bit, cols a multiple of 8) read or written in boxes of 64 columns x
// 1 head x box_tok tokens.  Head dimensions below 128 are described with their own column count, so boxes at
// columns >= cols load zeros (the kernels' tiles are 128 columns wide) and stores clip there.
inline bool make_token_map(CUtensorMap *map, const void *base, bool bf16, int cols, int heads, uint64_t tokens,
                           uint32_t box_tok) {
    return make_tmap_3d(map, base, bf16, (uint64_t)cols, (uint64_t)heads, tokens, (uint64_t)cols * 2,
                        (uint64_t)heads * cols * 2, 64, 1, box_tok);
}

}  // namespace gdr
