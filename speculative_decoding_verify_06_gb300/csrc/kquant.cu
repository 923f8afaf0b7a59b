// kquant.cu -- the verify GEMM on K-quant (Q4_K) super-block weights, read in their own layout.
//
// "100 tokens per second from a 27B model on a 24 GB AMD card", section "The wall", and "Decode
// is memory-bound ...", section "The ceiling": the pages' 27B checkpoints are UD-Q4_K_XL and
// Q4_K_M mixes whose 4-bit tensors are Q4_K super-blocks.  The pages give no layout; this file
// reads the format's public specification: 256 weights of one row per 144-byte super-block --
// fp16 d, fp16 dmin, 12 bytes of packed 6-bit sub-block scales sc[j] and mins m[j] (one pair
// per 32 weights), 128 bytes of 4-bit codes (byte 32 g + l holds weight 64 g + l in its low
// nibble and 64 g + 32 + l in its high nibble) -- and weight value d sc[j] q - dmin m[j].
//
//     Y[c][r] = sum_j ( d sc[j] * sum_{i in j} q_i x[c][i]  -  dmin m[j] * sum_{i in j} x[c][i] )
//
// A CUDA-core kernel: a CTA takes 32 rows at a time (4 per warp) and walks the inputs in tiles
// of 2048, staging each tile of the activations in shared memory as fp32 (one pad word per 32
// inputs, so the lanes' sub-blocks fall on different banks) together with each sub-block's
// activation sum; lane l of a warp takes sub-blocks l and l + 32 of the tile for each of the
// warp's rows, decodes the sub-block's (sc, m) from its super-block's header, builds the codes
// exactly as fp32 (2^23 + q minus 2^23) and accumulates the sub-block's dot product per column
// in fp32, then adds d sc * dot - dmin m * sum (d sc and dmin m are exact in fp32).  The warp
// sums its lanes with shuffles at the end of the row group.
#include "svd_common.cuh"

namespace svd {

constexpr int kKqThreads = 256;
constexpr int kKqRowsPerWarp = 4;
constexpr int kKqRows = (kKqThreads / 32) * kKqRowsPerWarp;  // rows per CTA pass
constexpr int kKqTile = 2048;                                // inputs per staged tile
constexpr int kKqPitch = kKqTile + kKqTile / 32;             // padded floats per column
constexpr int kKqBlockBytes = 144;                           // one super-block of 256 weights

template <int CC>
__global__ void __launch_bounds__(kKqThreads)
vl_q4k_kernel(const uint8_t *__restrict__ blocks, const __nv_bfloat16 *__restrict__ X,
              float *__restrict__ Y, int64_t in_f, int64_t out_f) {
    extern __shared__ float kq_smem[];
    float *xs = kq_smem;                        // [CC][kKqPitch]
    float *xsum = kq_smem + CC * kKqPitch;      // [CC][kKqTile / 32]
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row_bytes = in_f / 256 * kKqBlockBytes;
    for (int64_t r0 = (int64_t)blockIdx.x * kKqRows; r0 < out_f; r0 += (int64_t)gridDim.x * kKqRows) {
        float acc[kKqRowsPerWarp][CC];
#pragma unroll
        for (int rr = 0; rr < kKqRowsPerWarp; ++rr)
#pragma unroll
            for (int c = 0; c < CC; ++c) acc[rr][c] = 0.f;
        for (int64_t k0 = 0; k0 < in_f; k0 += kKqTile) {
            const int kt = (int)min((int64_t)kKqTile, in_f - k0);  // a multiple of 256
            const int nsub = kt / 32;
            __syncthreads();  // the previous tile is no longer read
            for (int i = threadIdx.x; i < CC * kt; i += kKqThreads) {
                const int c = i / kt, k = i - c * kt;
                xs[c * kKqPitch + k + k / 32] = __bfloat162float(X[(int64_t)c * in_f + k0 + k]);
            }
            __syncthreads();
            for (int i = threadIdx.x; i < CC * nsub; i += kKqThreads) {
                const int c = i / nsub, s = i - c * nsub;
                const float *xb = xs + c * kKqPitch + s * 33;
                float t = 0.f;
                for (int u = 0; u < 32; ++u) t += xb[u];
                xsum[c * (kKqTile / 32) + s] = t;
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < kKqRowsPerWarp; ++rr) {
                const int64_t row = r0 + warp * kKqRowsPerWarp + rr;
                if (row >= out_f) break;
                const uint8_t *rb = blocks + row * row_bytes + (k0 / 256) * kKqBlockBytes;
                for (int s = lane; s < nsub; s += 32) {
                    const int j = s & 7;
                    const uint8_t *blk = rb + (s >> 3) * kKqBlockBytes;
                    // header: d, dmin (bytes 0..3), scale bytes s0..s11 (bytes 4..15)
                    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
                    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
                    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                    int sc, m;
                    if (j < 4) {
                        sc = (int)((h.y >> (8 * j)) & 63u);
                        m = (int)((h.z >> (8 * j)) & 63u);
                    } else {
                        const int jj = j - 4;
                        const unsigned lo = (h.w >> (8 * jj)) & 255u;
                        sc = (int)((lo & 15u) | (((h.y >> (8 * jj + 6)) & 3u) << 4));
                        m = (int)((lo >> 4) | (((h.z >> (8 * jj + 6)) & 3u) << 4));
                    }
                    const float a = d * (float)sc, bm = dmin * (float)m;
                    // codes of sub-block j: bytes 32 (j / 2) .. + 31, low nibbles for even j
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * (j >> 1));
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * (j >> 1) + 16);
                    const uint32_t wds[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    const int sh = (j & 1) * 4;
                    float dot[CC];
#pragma unroll
                    for (int c = 0; c < CC; ++c) dot[c] = 0.f;
                    const float *xb = xs + s * 33;
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi)
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            const uint32_t qv = (wds[wi] >> (8 * n + sh)) & 15u;
                            const float qf = __uint_as_float(0x4B000000u | qv) - 8388608.0f;
#pragma unroll
                            for (int c = 0; c < CC; ++c) dot[c] = fmaf(qf, xb[c * kKqPitch + 4 * wi + n], dot[c]);
                        }
#pragma unroll
                    for (int c = 0; c < CC; ++c)
                        acc[rr][c] = fmaf(a, dot[c], fmaf(-bm, xsum[c * (kKqTile / 32) + s], acc[rr][c]));
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < kKqRowsPerWarp; ++rr) {
            const int64_t row = r0 + warp * kKqRowsPerWarp + rr;
#pragma unroll
            for (int c = 0; c < CC; ++c) {
                float v = acc[rr][c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0 && row < out_f) Y[(int64_t)c * out_f + row] = v;
            }
        }
    }
}

template <int CC>
static cudaError_t launch_q4k(const svd_qweight *W, const void *X, float *Y, bool pdl,
                              cudaStream_t stream) {
    auto kern = vl_q4k_kernel<CC>;
    const size_t smem = (size_t)CC * (kKqPitch + kKqTile / 32) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kKqThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    const int64_t need = (W->out_features + kKqRows - 1) / kKqRows;
    if (grid > need) grid = need;
    return launch(kern, dim3((unsigned)grid), dim3(kKqThreads), smem, stream, pdl,
                  reinterpret_cast<const uint8_t *>(W->codes),
                  reinterpret_cast<const __nv_bfloat16 *>(X), Y, W->in_features, W->out_features);
}

// Y = W x for a Q4_K matrix; C in 1..8 (checked by the caller), in_features % 256 == 0.
int verify_linear_q4k(const svd_qweight *W, const void *X, int C, float *Y, bool pdl,
                      cudaStream_t stream) {
    cudaError_t e;
    switch (C) {
        case 1: e = launch_q4k<1>(W, X, Y, pdl, stream); break;
        case 2: e = launch_q4k<2>(W, X, Y, pdl, stream); break;
        case 3: e = launch_q4k<3>(W, X, Y, pdl, stream); break;
        case 4: e = launch_q4k<4>(W, X, Y, pdl, stream); break;
        case 5: e = launch_q4k<5>(W, X, Y, pdl, stream); break;
        case 6: e = launch_q4k<6>(W, X, Y, pdl, stream); break;
        case 7: e = launch_q4k<7>(W, X, Y, pdl, stream); break;
        case 8: e = launch_q4k<8>(W, X, Y, pdl, stream); break;
        default: return SVD_ERR_UNSUPPORTED;
    }
    SVD_CUDA_TRY(e);
    return SVD_OK;
}

}  // namespace svd
