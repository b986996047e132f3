// qmv_generic.cu -- the exact-but-plain kernels: the matrix-vector fallback for
// shapes or alignments the streaming kernel does not take (K % 256 != 0, or a
// weight pointer not 16-byte aligned) and for Q4_K off the tensor-core path,
// the whole-matrix dequantizers and the token-table row gather.
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"

namespace qbw {
namespace {

template <int FMT>
__device__ __forceinline__ float code_at(const uint8_t* blk, int k) {
    if constexpr (FMT == kFmtQ8) {
        return (float)(int)(int8_t)blk[2 + k];
    } else {
        const uint32_t byte = blk[2 + (k & 15)];
        const uint32_t code = (k < 16) ? (byte & 0x0Fu) : (byte >> 4);
        return (float)((int)code - 8);
    }
}

// One warp per output row; lane l takes blocks l, l+32, ...; byte loads only.
template <int FMT, int NMAT>
__global__ void __launch_bounds__(256) qmv_generic_kernel(const uint8_t* w0, const uint8_t* w1, const void* x,
                                                          int x_bf16, void* y, int y_bf16, int64_t N, int64_t K) {
    constexpr int BPB = (FMT == kFmtQ4) ? 18 : 34;
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32;
    const int64_t row_bytes = nb * BPB;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); n < N; n += warps) {
        float acc[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) acc[m] = 0.f;
        for (int64_t b = lane; b < nb; b += 32) {
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const uint8_t* blk = ((m == 0) ? w0 : w1) + n * row_bytes + b * BPB;
                const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
                float s = 0.f;
                for (int k = 0; k < 32; ++k) {
                    const int64_t i = b * 32 + k;
                    const float xv = x_bf16 ? load_act<__nv_bfloat16>(x, i) : load_act<float>(x, i);
                    s = fmaf(code_at<FMT>(blk, k), xv, s);
                }
                acc[m] = fmaf(d, s, acc[m]);
            }
        }
        float v = 0.f;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            float t = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            acc[m] = t;
        }
        v = acc[0];
        if constexpr (NMAT == 2) v = gelu_tanh(acc[0]) * acc[1];
        if (lane == 0) {
            if (y_bf16) store_out<__nv_bfloat16>(y, n, v);
            else store_out<float>(y, n, v);
        }
    }
}

// ---------------------------------------------------------------- Q4_K
// A Q4_K super-block (GGUF block_q4_K, 144 bytes, 256 weights): fp16 d at
// byte 0, fp16 dmin at byte 2, 12 scale bytes s[] at byte 4, 128 nibble bytes
// at byte 16.  Sub-block j (32 weights) has a six-bit scale sc_j and min m_j:
// for j < 4 the low six bits of s[j] and s[j + 4]; for j >= 4 the low and high
// nibble of s[j + 4], with the top two bits taken from s[j - 4] (sc) and s[j]
// (m).  Weight e = 64 i + l (chunk i) has code (l < 32 ? low : high) nibble of
// byte 32 i + (l % 32).  w = d sc_j q - dmin m_j (jouleclaw-loader-gguf
// BENCHMARKS, "Q4_K matmul -- scalar fused vs AMX-tiled").
__device__ __forceinline__ void q4k_sub_scale(const uint8_t* s, int j, int& sc, int& m) {
    if (j < 4) {
        sc = s[j] & 63;
        m = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

__device__ __forceinline__ int q4k_code_at(const uint8_t* qs, int e) {
    const uint32_t byte = qs[32 * (e >> 6) + (e & 31)];
    return (e & 32) ? (int)(byte >> 4) : (int)(byte & 15u);
}

// One warp per output row; lane l takes super-blocks l, l + 32, ...  Per
// sub-block the algebraic split: d sc_j * sum(q x) - dmin m_j * sum(x).
__global__ void __launch_bounds__(256) qmv_q4k_generic_kernel(const uint8_t* w, const void* x, int x_bf16, void* y,
                                                              int y_bf16, int64_t N, int64_t K) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 256;
    const int64_t row_bytes = nb * 144;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); n < N; n += warps) {
        float acc = 0.f;
        for (int64_t b = lane; b < nb; b += 32) {
            const uint8_t* blk = w + n * row_bytes + b * 144;
            const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
            const float dmin = half_bits_to_float((uint32_t)blk[2] | ((uint32_t)blk[3] << 8));
            for (int j = 0; j < 8; ++j) {
                int sc, m;
                q4k_sub_scale(blk + 4, j, sc, m);
                float s1 = 0.f, s0 = 0.f;
                for (int t = 0; t < 32; ++t) {
                    const int e = 32 * j + t;
                    const int64_t i = b * 256 + e;
                    const float xv = x_bf16 ? load_act<__nv_bfloat16>(x, i) : load_act<float>(x, i);
                    s1 = fmaf((float)q4k_code_at(blk + 16, e), xv, s1);
                    s0 += xv;
                }
                acc = fmaf(d * (float)sc, s1, acc);
                acc = fmaf(-dmin * (float)m, s0, acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (y_bf16) store_out<__nv_bfloat16>(y, n, acc);
            else store_out<float>(y, n, acc);
        }
    }
}

// One thread per super-block: w = (d sc) q - dmin m.  d sc, (d sc) q and
// dmin m are exact in fp32 (at most 21 significant bits), so the single
// rounding of the difference gives the nearest fp32 to the exact weight.
__global__ void __launch_bounds__(256) dequant_q4k_kernel(const uint8_t* w, float* out, int64_t N, int64_t K) {
    const int64_t nb = K / 256;
    const int64_t total = N * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t* blk = w + i * 144;
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        const float dmin = half_bits_to_float((uint32_t)blk[2] | ((uint32_t)blk[3] << 8));
        const int64_t n = i / nb, b = i - n * nb;
        float* o = out + n * K + b * 256;
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            q4k_sub_scale(blk + 4, j, sc, m);
            const float ds = __fmul_rn(d, (float)sc), dm = __fmul_rn(dmin, (float)m);
#pragma unroll 8
            for (int t = 0; t < 32; ++t) o[32 * j + t] = __fsub_rn(__fmul_rn(ds, (float)q4k_code_at(blk + 16, 32 * j + t)), dm);
        }
    }
}

// One thread per block: out[n*K + 32b + k] = d * code (exact in fp32).
template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* w, float* out, int64_t N, int64_t K) {
    constexpr int BPB = (FMT == kFmtQ4) ? 18 : 34;
    const int64_t nb = K / 32;
    const int64_t total = N * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t* blk = w + i * BPB;
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        const int64_t n = i / nb, b = i - n * nb;
        float* o = out + n * K + b * 32;
#pragma unroll 8
        for (int k = 0; k < 32; ++k) o[k] = d * code_at<FMT>(blk, k);
    }
}

// Token-table gather: one thread per (output row, block, 8 consecutive
// elements); out[i, 32b + k] = d * q of block b of row ids[i], exact in fp32
// (bf16: rounded to nearest even).  An index outside [0, N) gives zeros and
// fault code 3.
template <int FMT, typename T>
__global__ void __launch_bounds__(256) embed_kernel(const uint8_t* w, const int32_t* ids, int64_t n_ids, int64_t N,
                                                    int64_t K, T* out, unsigned int* fault) {
    constexpr int BPB = (FMT == kFmtQ4) ? 18 : 34;
    const int64_t nb = K / 32;
    const int64_t total = n_ids * nb * 4;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t ib = t >> 2;                 // (row, block)
        const int k0 = (int)(t & 3) * 8;           // first of this thread's 8 elements
        const int64_t i = ib / nb, b = ib - i * nb;
        const int64_t id = ids[i];
        T* o = out + i * K + b * 32 + k0;
        float v[8];
        if (id < 0 || id >= N) {
            if (k0 == 0) record_fault(fault, kFaultBadIndex);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = 0.f;
        } else {
            const uint8_t* blk = w + (id * nb + b) * BPB;
            const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = d * code_at<FMT>(blk, k0 + k);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) store_out<T>(o, k, v[k]);
    }
}

// Small-M fallback: one warp per weight row, X rows in groups of 8, exact
// codes times bf16 activations in fp32, scale applied per block.
__global__ void __launch_bounds__(256) qmm_generic_kernel(const uint8_t* w, const void* X, void* Y, int y_bf16,
                                                          int64_t M, int64_t N, int64_t K) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32;
    const int64_t row_bytes = nb * 18;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); n < N; n += warps) {
        for (int64_t m0 = 0; m0 < M; m0 += 8) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            for (int64_t b = lane; b < nb; b += 32) {
                const uint8_t* blk = w + n * row_bytes + b * 18;
                const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
                float s[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) s[i] = 0.f;
                for (int k = 0; k < 32; ++k) {
                    const float c = code_at<kFmtQ4>(blk, k);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (m0 + i < M) s[i] = fmaf(c, load_act<__nv_bfloat16>(X, (m0 + i) * K + b * 32 + k), s[i]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(d, s[i], acc[i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float t = acc[i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0 && m0 + i < M) {
                    if (y_bf16) store_out<__nv_bfloat16>(Y, (m0 + i) * N + n, t);
                    else store_out<float>(Y, (m0 + i) * N + n, t);
                }
            }
        }
    }
}

}  // namespace

// Self-test of the bounded waits: one thread waits, with a short limit, on
// something nothing will complete -- which = 0: phase 0 of a fresh mbarrier
// (the wait every pipeline stage uses; fault code 1), which = 1: the tag of a
// global word that stays 0 (the split-tile share wait; fault code 4).  The
// wait runs out, records its code in the fault word and the kernel returns.
__device__ unsigned long long g_selftest_word = 0ull;

__global__ void selftest_wait_kernel(int which, uint64_t limit_ns, unsigned int* fault) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        fence_mbar_init();
        mbar_wait_bounded(b, 0u, fault, kFaultBulkWaitTimeout, limit_ns);
    } else {
        wait_tag_u64(&g_selftest_word, launch_tag(), fault, kFaultShareWaitTimeout, limit_ns);   // stays 0
    }
}

cudaError_t launch_selftest_wait(int which, uint64_t limit_ns, unsigned int* fault, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(which, limit_ns, fault);
    return cudaGetLastError();
}

cudaError_t launch_qmm_generic(const uint8_t* w, const void* X, void* Y, int y_bf16, int64_t M, int64_t N,
                               int64_t K, int sm_count, cudaStream_t stream) {
    const int64_t want = (N + 7) / 8;
    const int ctas = (int)(want < (int64_t)sm_count * 8 ? want : (int64_t)sm_count * 8);
    qmm_generic_kernel<<<ctas, 256, 0, stream>>>(w, X, Y, y_bf16, M, N, K);
    return cudaGetLastError();
}

cudaError_t launch_qmv_generic(int fmt, int nmat, const uint8_t* w0, const uint8_t* w1, const void* x,
                               int x_bf16, void* y, int y_bf16, int64_t N, int64_t K, int sm_count,
                               cudaStream_t stream) {
    const int threads = 256;
    const int64_t want = (N + 7) / 8;
    const int ctas = (int)(want < (int64_t)sm_count * 8 ? want : (int64_t)sm_count * 8);
    if (fmt == kFmtQ4K)
        qmv_q4k_generic_kernel<<<ctas, threads, 0, stream>>>(w0, x, x_bf16, y, y_bf16, N, K);
    else if (fmt == kFmtQ8)
        qmv_generic_kernel<kFmtQ8, 1><<<ctas, threads, 0, stream>>>(w0, w1, x, x_bf16, y, y_bf16, N, K);
    else if (nmat == 1)
        qmv_generic_kernel<kFmtQ4, 1><<<ctas, threads, 0, stream>>>(w0, w1, x, x_bf16, y, y_bf16, N, K);
    else
        qmv_generic_kernel<kFmtQ4, 2><<<ctas, threads, 0, stream>>>(w0, w1, x, x_bf16, y, y_bf16, N, K);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* w, float* out, int64_t N, int64_t K, int sm_count,
                           cudaStream_t stream) {
    const int threads = 256;
    const int64_t blocks = N * (K / (fmt == kFmtQ4K ? 256 : 32));
    const int64_t want = (blocks + threads - 1) / threads;
    const int ctas = (int)(want < (int64_t)sm_count * 16 ? want : (int64_t)sm_count * 16);
    if (fmt == kFmtQ4K)
        dequant_q4k_kernel<<<ctas, threads, 0, stream>>>(w, out, N, K);
    else if (fmt == kFmtQ8)
        dequant_kernel<kFmtQ8><<<ctas, threads, 0, stream>>>(w, out, N, K);
    else
        dequant_kernel<kFmtQ4><<<ctas, threads, 0, stream>>>(w, out, N, K);
    return cudaGetLastError();
}

cudaError_t launch_embed(int fmt, const uint8_t* w, const int32_t* ids, int64_t n_ids, int64_t N, int64_t K, void* out,
                         int out_bf16, unsigned int* fault, int sm_count, cudaStream_t stream) {
    const int threads = 256;
    const int64_t items = n_ids * (K / 32) * 4;
    const int64_t want = (items + threads - 1) / threads;
    const int ctas = (int)(want < (int64_t)sm_count * 8 ? want : (int64_t)sm_count * 8);
    if (fmt == kFmtQ8) {
        if (out_bf16)
            embed_kernel<kFmtQ8, __nv_bfloat16>
                <<<ctas, threads, 0, stream>>>(w, ids, n_ids, N, K, static_cast<__nv_bfloat16*>(out), fault);
        else
            embed_kernel<kFmtQ8, float><<<ctas, threads, 0, stream>>>(w, ids, n_ids, N, K, static_cast<float*>(out), fault);
    } else {
        if (out_bf16)
            embed_kernel<kFmtQ4, __nv_bfloat16>
                <<<ctas, threads, 0, stream>>>(w, ids, n_ids, N, K, static_cast<__nv_bfloat16*>(out), fault);
        else
            embed_kernel<kFmtQ4, float><<<ctas, threads, 0, stream>>>(w, ids, n_ids, N, K, static_cast<float*>(out), fault);
    }
    return cudaGetLastError();
}

}  // namespace qbw
