// quantize.h -- internal interface of the MX quantiser kernel (quantize.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace mxg {

constexpr int kQuantFmtMxfp8 = 1;
constexpr int kQuantFmtMxfp4 = 2;
constexpr int kQuantInF32 = 1;
constexpr int kQuantInBf16 = 2;

struct QuantParams {
    const void *x;     // rows x K input, row-major, 16-byte aligned
    void *codes;       // rows x K (MXFP8) or rows x K/2 (MXFP4) bytes
    uint8_t *scales;   // rows x K/32 row-major, or the tile layout when tiled
    int64_t rows;
    int64_t K;         // multiple of 32 (of 128 when tiled)
    int fmt;           // kQuantFmt*
    int in_dtype;      // kQuantIn*
    int tiled;         // 1: scales in the 512-byte tile layout (rows padded to 128)
    int sf_words;      // row-major scales written as 4-byte words (K % 128 == 0)
};

// Validated arguments only (the C ABI checks them).
cudaError_t launch_quantize(const QuantParams &p, int num_sms, cudaStream_t s);

}  // namespace mxg
