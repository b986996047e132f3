// qmv_mixbit.cu -- y = W x for the mixed-bit matrices of a QAT checkpoint:
// int2-symmetric, int4-affine and int8 (Core AI model zoo, Gemma-4-E2B
// raw-Metal port, "What shipped": mixed-bit matvecs over quantized words qp,
// scales sc and biases bi).  Layout (include/qbw.h): fields of b bits packed
// lowest bits first into 32-bit words, rows back to back; one fp16 scale (and,
// for int4, one fp16 bias) per group of G weights of a row.
//   b = 2: q = two's-complement field (-2 .. 1), w = sc q
//   b = 4: c = unsigned field (0 .. 15),       w = sc c + bi
//   b = 8: q = two's-complement byte,           w = sc q
//
// One token, bandwidth-bound.  A CTA stages x once as fp32 in shared memory
// (XOR-swizzled so that each lane's 16-byte reads of its chunk are free of
// bank conflicts), and for int4 the sum of x over every 32-bit word's
// elements (the bias term of the split sc * sum(c x) + bi * sum(x)).  A warp
// takes R rows at a time; lane l streams 16-byte word groups l, l + 32, ... of
// each row (coalesced), turns each field into an exact float with one byte
// permute against 2^23 and a packed subtract, and accumulates per word with
// packed fp32x2 FMAs; the word's sum is scaled by its group's sc (plus bi times
// the word's sum of x) in fp32.  The rows' sums are reduced across the warp in
// a fixed order, so results are bit-reproducible.
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"

namespace qbw {
namespace {

constexpr int kMixThreads = 256;

struct MixParams {
    const uint4* qp;        // [N][wq] word groups
    const uint16_t* sc;     // [N][K / G] fp16 bits
    const uint16_t* bi;     // [N][K / G] fp16 bits (4-bit only)
    const void* x;          // [K] fp32 or bf16
    void* y;                // [N] fp32 or bf16
    int32_t N, K, G, wq;    // wq = 16-byte word groups per row
    int32_t gshift;         // log2 G when G is a power of two, else -1
    int32_t x_bf16, y_bf16;
};

// The scale group of element e of a row: e / G (a shift when G is a power of two)
__device__ __forceinline__ int group_of(const MixParams& p, int e) { return p.gshift >= 0 ? e >> p.gshift : e / p.G; }

// Elements of a 16-byte word group and of a 32-bit word, for b-bit fields.
template <int BITS> constexpr int kElems = 128 / BITS;
template <int BITS> constexpr int kWordElems = 32 / BITS;

// Float4 slot, in the staged x, of float4 j of chunk ch (chunk = one word
// group's elements): XOR-swizzled within the chunk.
template <int BITS>
__device__ __forceinline__ int x_slot(int ch, int j) {
    constexpr int F = kElems<BITS> / 4;                 // float4 per chunk: 16, 8, 4
    constexpr int SW = F < 8 ? F - 1 : 7;
    return ch * F + (j ^ (ch & SW));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Byte k of v as the float 2^23 + byte (the byte in the low mantissa bits).
template <int K>
__device__ __forceinline__ uint32_t byte_magic(uint32_t v) {
    return prmt(v, 0x4B000000u, 0x7540u | (uint32_t)K);
}

// acc (two fp32 lanes) += (f - m) * x, f two magic floats, m the magic
// offset: the subtraction is exact, the products and sums round in fp32.
__device__ __forceinline__ void fma_pair(uint64_t& acc, uint32_t f0, uint32_t f1, uint64_t m, float x0, float x1) {
    const uint64_t c = fadd2(pack2(f0, f1), m);
    ffma2(acc, c, pack2f(x0, x1));
}

// acc (two fp32 partial sums) += the dot product of one 32-bit word's fields
// with their activations xw[] (kWordElems<BITS> of them, in element order).
template <int BITS>
__device__ __forceinline__ void word_dot(uint64_t& acc, uint32_t w, const float* xw) {
    if constexpr (BITS == 8) {
        // q + 128 in each byte, then 2^23 + q + 128 - (2^23 + 128) = q
        const uint32_t u = w ^ 0x80808080u;
        const uint64_t m = pack2f(-8388736.f, -8388736.f);
        fma_pair(acc, byte_magic<0>(u), byte_magic<1>(u), m, xw[0], xw[1]);
        fma_pair(acc, byte_magic<2>(u), byte_magic<3>(u), m, xw[2], xw[3]);
    } else if constexpr (BITS == 4) {
        // even elements in the low nibbles, odd ones in the high nibbles
        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        const uint64_t m = pack2f(-8388608.f, -8388608.f);
        fma_pair(acc, byte_magic<0>(lo), byte_magic<0>(hi), m, xw[0], xw[1]);
        fma_pair(acc, byte_magic<1>(lo), byte_magic<1>(hi), m, xw[2], xw[3]);
        fma_pair(acc, byte_magic<2>(lo), byte_magic<2>(hi), m, xw[4], xw[5]);
        fma_pair(acc, byte_magic<3>(lo), byte_magic<3>(hi), m, xw[6], xw[7]);
    } else {
        // field 4k + s in byte k of t_s; (f ^ 2) - 2 is the two's-complement value
        uint32_t t[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) t[s] = ((w >> (2 * s)) & 0x03030303u) ^ 0x02020202u;
        const uint64_t m = pack2f(-8388610.f, -8388610.f);
        fma_pair(acc, byte_magic<0>(t[0]), byte_magic<0>(t[1]), m, xw[0], xw[1]);
        fma_pair(acc, byte_magic<0>(t[2]), byte_magic<0>(t[3]), m, xw[2], xw[3]);
        fma_pair(acc, byte_magic<1>(t[0]), byte_magic<1>(t[1]), m, xw[4], xw[5]);
        fma_pair(acc, byte_magic<1>(t[2]), byte_magic<1>(t[3]), m, xw[6], xw[7]);
        fma_pair(acc, byte_magic<2>(t[0]), byte_magic<2>(t[1]), m, xw[8], xw[9]);
        fma_pair(acc, byte_magic<2>(t[2]), byte_magic<2>(t[3]), m, xw[10], xw[11]);
        fma_pair(acc, byte_magic<3>(t[0]), byte_magic<3>(t[1]), m, xw[12], xw[13]);
        fma_pair(acc, byte_magic<3>(t[2]), byte_magic<3>(t[3]), m, xw[14], xw[15]);
    }
}

__device__ __forceinline__ float half_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ uint4 ld_shared16(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool live) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(live ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool live) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(live ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Each lane streams its own 16-byte word groups (one per row of the warp's
// item of ROWS rows) and the 4-byte words that hold their scales (and
// biases) through a ring of STAGES stages in shared memory, with cp.async:
// STAGES - 1 steps are in flight while it computes one.  A lane reads back
// only what it copied itself.  Two shapes of the ring (mix_shape): 4 rows
// and 3 stages for 4- and 8-bit matrices of K <= 8192 (the activations a row
// item shares are read once for 4 rows), else 2 rows and 4 stages (smaller
// rings beside long activation vectors, more CTAs per SM).
struct MixShape {
    int rows, stages;
};
__host__ __device__ constexpr MixShape mix_shape(int bits, int64_t K) {
    return (bits >= 4 && K <= 8192) ? MixShape{4, 3} : MixShape{2, 4};
}

// Scale groups per 16-byte word group: 1 when a group covers it, else E / G.
template <int BITS, int SW, int ROWS, int STAGES>
struct MixRing {
    // [stage][row][lane] word groups, then [stage][row][sw][lane] scale words
    // (and bias words for 4 bits)
    static constexpr uint32_t kQBytes = STAGES * ROWS * 32 * 16;
    static constexpr uint32_t kSBytes = STAGES * ROWS * SW * 32 * 4;
    static constexpr uint32_t kWarpBytes = kQBytes + kSBytes * (BITS == 4 ? 2 : 1);
    __device__ static uint32_t q(uint32_t base, int st, int r, int lane) {
        return base + (uint32_t)(((st * ROWS + r) * 32 + lane) * 16);
    }
    __device__ static uint32_t sc(uint32_t base, int st, int r, int k, int lane) {
        return base + kQBytes + (uint32_t)((((st * ROWS + r) * SW + k) * 32 + lane) * 4);
    }
    __device__ static uint32_t bi(uint32_t base, int st, int r, int k, int lane) {
        return sc(base, st, r, k, lane) + kSBytes;
    }
};

// A step of a warp: item `it` (rows it * ROWS ..), word group c of each
// row, in ring stage st.
template <int BITS, int SW, int ROWS, int STAGES>
__device__ __forceinline__ void issue_step(const MixParams& p, uint32_t ring, int st, int it, int c, int items,
                                           int gpr, int lane) {
    using R = MixRing<BITS, SW, ROWS, STAGES>;
    constexpr int E = kElems<BITS>;
    const int n0 = it * ROWS;
    const int g0 = c < p.wq ? group_of(p, c * E) : 0;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const bool live = it < items && n0 + r < p.N && c < p.wq;
        const size_t row = live ? (size_t)(n0 + r) : 0;
        cp_async16(R::q(ring, st, r, lane), p.qp + row * p.wq + (live ? c : 0), live);
#pragma unroll
        for (int k = 0; k < SW; ++k) {
            // the 4-byte word holding scale element (row, group) (sc, bi 4-byte aligned)
            const size_t e = live ? row * gpr + (size_t)(g0 + k) : 0;
            cp_async4(R::sc(ring, st, r, k, lane), p.sc + (e & ~size_t(1)), live);
            if constexpr (BITS == 4) cp_async4(R::bi(ring, st, r, k, lane), p.bi + (e & ~size_t(1)), live);
        }
    }
}

// A warp's step cursor: item index j (item warp + j * nwarps) and step cs
// within the item (word group lane + 32 cs), advanced without divisions.
struct MixCursor {
    int j = 0, cs = 0;
    __device__ void next(int S) {
        if (++cs == S) {
            cs = 0;
            ++j;
        }
    }
};

// fp16 half (e & 1) of the 4-byte word at shared address a, as float
__device__ __forceinline__ float ring_half(uint32_t a, uint32_t odd) {
    const uint32_t w = lds32(a);
    return half_to_float((uint16_t)(odd ? (w >> 16) : (w & 0xFFFFu)));
}

// Dynamic shared memory: x as fp32 in swizzled chunks [K], (4-bit) the per-word
// sums of x [K / 8], then each warp's ring.
template <int BITS, int SW, int ROWS, int STAGES>
__global__ void __launch_bounds__(kMixThreads) qmv_mixbit_kernel(const __grid_constant__ MixParams p) {
    using R = MixRing<BITS, SW, ROWS, STAGES>;
    extern __shared__ __align__(16) float xs[];
    float* xw_sum = xs + p.K;
    constexpr int E = kElems<BITS>, EW = kWordElems<BITS>;
    const int lane = threadIdx.x & 31;
    const int warp = (int)(blockIdx.x * (kMixThreads / 32) + (threadIdx.x >> 5));
    const int nwarps = (int)(gridDim.x * (kMixThreads / 32));
    const int items = (p.N + ROWS - 1) / ROWS;
    const int gpr = p.K / p.G;                           // groups per row
    const int S = (p.wq + 31) / 32;                      // steps per item
    const int my_items = warp < items ? (items - warp + nwarps - 1) / nwarps : 0;
    const int T = my_items * S;                          // this warp's steps
    const uint32_t xbytes = (uint32_t)p.K * 4u + (BITS == 4 ? (uint32_t)(p.K / 8) * 4u : 0u);
    const uint32_t ring = smem_u32(xs) + ((xbytes + 127u) & ~127u) + (uint32_t)(threadIdx.x >> 5) * R::kWarpBytes;
    // the weights do not depend on the preceding grid: the first steps are
    // issued before the activations are waited for and staged
    MixCursor iss;
#pragma unroll
    for (int t = 0; t < STAGES - 1; ++t) {
        if (t < T)
            issue_step<BITS, SW, ROWS, STAGES>(p, ring, t, warp + iss.j * nwarps, lane + 32 * iss.cs, items, gpr, lane);
        iss.next(S);
        cp_async_commit();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    // stage x: float4 f of the vector is float4 f % (E / 4) of chunk f / (E / 4)
    for (int f = threadIdx.x; f < p.K / 4; f += kMixThreads) {
        float4 v;
        if (p.x_bf16) {
            const uint2 b = __ldg(reinterpret_cast<const uint2*>(p.x) + f);
            v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u), __uint_as_float(b.y << 16),
                            __uint_as_float(b.y & 0xFFFF0000u));
        } else {
            v = __ldg(reinterpret_cast<const float4*>(p.x) + f);
        }
        reinterpret_cast<float4*>(xs)[x_slot<BITS>(f / (E / 4), f % (E / 4))] = v;
    }
    __syncthreads();
    if constexpr (BITS == 4) {
        // sum of x over each 32-bit word's 8 elements (element order), then
        // over each scale group's words of a word group: xw_sum[ch * SW + k]
        // (words kept in order, pairwise within the group)
        for (int sg = threadIdx.x; sg < (p.K / E) * SW; sg += kMixThreads) {
            const int ch = sg / SW, k = sg % SW;
            float tot = 0.f;
#pragma unroll
            for (int wi = 0; wi < 4 / SW; ++wi) {
                const int j = 2 * (k * (4 / SW) + wi);
                const float4 a = reinterpret_cast<const float4*>(xs)[x_slot<BITS>(ch, j)];
                const float4 b = reinterpret_cast<const float4*>(xs)[x_slot<BITS>(ch, j + 1)];
                tot += ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            }
            xw_sum[sg] = tot;
        }
        __syncthreads();
    }
    float acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
    MixCursor cur;
    int st = 0, ist = STAGES - 1;                  // stages of the step consumed and issued next
    for (int t = 0; t < T; ++t) {
        // step t + STAGES - 1 into the stage step t - 1 has freed
        if (t + STAGES - 1 < T)
            issue_step<BITS, SW, ROWS, STAGES>(p, ring, ist, warp + iss.j * nwarps, lane + 32 * iss.cs, items, gpr,
                                               lane);
        iss.next(S);
        ist = ist + 1 == STAGES ? 0 : ist + 1;
        cp_async_commit();
        cp_async_wait<STAGES - 1>();              // step t's copies have landed
        const int c = lane + 32 * cur.cs;
        const int n0 = (warp + cur.j * nwarps) * ROWS;
        if (c < p.wq) {
            const int g0 = group_of(p, c * E);
            uint4 q[ROWS];
            uint64_t dot[ROWS][SW];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                q[r] = ld_shared16(R::q(ring, st, r, lane));
#pragma unroll
                for (int k = 0; k < SW; ++k) dot[r][k] = 0ull;
            }
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                // the word's activations: EW floats, float4 slots of chunk c
                float xv[EW];
#pragma unroll
                for (int q4 = 0; q4 < EW / 4; ++q4) {
                    const float4 v = reinterpret_cast<const float4*>(xs)[x_slot<BITS>(c, wi * (EW / 4) + q4)];
                    xv[4 * q4] = v.x;
                    xv[4 * q4 + 1] = v.y;
                    xv[4 * q4 + 2] = v.z;
                    xv[4 * q4 + 3] = v.w;
                }
                constexpr int kWordsPerGroup = 4 / SW;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t w = wi == 0 ? q[r].x : wi == 1 ? q[r].y : wi == 2 ? q[r].z : q[r].w;
                    word_dot<BITS>(dot[r][wi / kWordsPerGroup], w, xv);
                }
            }
            // per scale group of the step: acc += sc * dot (+ bi * sum x); the
            // scale element's index parity picks its half of the copied word
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
#pragma unroll
                for (int k = 0; k < SW; ++k) {
                    const uint32_t odd = ((uint32_t)(n0 + r) * (uint32_t)gpr + (uint32_t)(g0 + k)) & 1u;
                    const float2 d = unpack2f(dot[r][k]);
                    acc[r] = fmaf(ring_half(R::sc(ring, st, r, k, lane), odd), d.x + d.y, acc[r]);
                    if constexpr (BITS == 4)
                        acc[r] = fmaf(ring_half(R::bi(ring, st, r, k, lane), odd), xw_sum[c * SW + k], acc[r]);
                }
            }
        }
        if (cur.cs == S - 1) {
            // the item's last step: reduce and store its rows
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
            }
            if (lane < ROWS && n0 + lane < p.N) {
                float v = acc[0];
#pragma unroll
                for (int r = 1; r < ROWS; ++r)
                    if (lane == r) v = acc[r];
                if (p.y_bf16) store_out<__nv_bfloat16>(p.y, n0 + lane, v);
                else store_out<float>(p.y, n0 + lane, v);
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
        }
        cur.next(S);
        st = st + 1 == STAGES ? 0 : st + 1;
    }
    cp_async_wait<0>();
}

// out[n * K + k] = w[n, k] in fp32: sc * q, or fmaf(sc, c, bi) (one rounding)
template <int BITS>
__global__ void dequant_mixbit_kernel(const uint32_t* qp, const uint16_t* sc, const uint16_t* bi, int G, int N, int K,
                                      float* out) {
    constexpr int EW = kWordElems<BITS>;
    const int64_t words = (int64_t)N * (K / EW);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / (K / EW), e0 = (i % (K / EW)) * EW;
        const int64_t gi = n * (K / G) + e0 / G;
        const float s = half_to_float(sc[gi]);
        const float b = BITS == 4 ? half_to_float(bi[gi]) : 0.f;
        const uint32_t w = qp[i];
#pragma unroll
        for (int e = 0; e < EW; ++e) {
            int v = (int)((w >> (e * BITS)) & ((1u << BITS) - 1u));
            if (BITS != 4 && v >= (1 << (BITS - 1))) v -= 1 << BITS;
            out[n * K + e0 + e] = BITS == 4 ? fmaf(s, (float)v, b) : s * (float)v;
        }
    }
}

template <int BITS, int SW, int ROWS, int STAGES>
cudaError_t launch_mix(const MixParams& p, int sm_count, cudaStream_t stream) {
    const size_t smem = qmv_mixbit_smem_bytes(BITS, p.K, p.G);
    static_assert(MixRing<BITS, SW, ROWS, STAGES>::kWarpBytes * (kMixThreads / 32) ==
                      (size_t)STAGES * ROWS * 32 * (16 + SW * 4 * (BITS == 4 ? 2 : 1)) * (kMixThreads / 32),
                  "ring size");
    static thread_local int prepared = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (prepared != dev) {
        cudaError_t e = cudaFuncSetAttribute(qmv_mixbit_kernel<BITS, SW, ROWS, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMixMaxSmem);
        if (e != cudaSuccess) return e;
        prepared = dev;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmv_mixbit_kernel<BITS, SW, ROWS, STAGES>, kMixThreads,
                                                                  smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int items = (p.N + ROWS - 1) / ROWS;
    const int warps_per_cta = kMixThreads / 32;
    int ctas = sm_count * per_sm;
    if (ctas * warps_per_cta > items) ctas = (items + warps_per_cta - 1) / warps_per_cta;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kMixThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmv_mixbit_kernel<BITS, SW, ROWS, STAGES>, p);
}

template <int BITS, int ROWS, int STAGES>
cudaError_t launch_mix_sw(const MixParams& p, int sm_count, cudaStream_t stream) {
    constexpr int E = kElems<BITS>;
    const int sw = p.G >= E ? 1 : E / p.G;
    if (sw == 1) return launch_mix<BITS, 1, ROWS, STAGES>(p, sm_count, stream);
    if constexpr (E >= 32) {
        if (sw == 2) return launch_mix<BITS, 2, ROWS, STAGES>(p, sm_count, stream);
    }
    if constexpr (E >= 64) {
        if (sw == 4) return launch_mix<BITS, 4, ROWS, STAGES>(p, sm_count, stream);
    }
    return cudaErrorInvalidValue;
}

template <int BITS>
cudaError_t launch_mix_shape(const MixParams& p, int sm_count, cudaStream_t stream) {
    if (mix_shape(BITS, p.K).rows == 4) {
        if constexpr (BITS >= 4) return launch_mix_sw<BITS, 4, 3>(p, sm_count, stream);
    }
    return launch_mix_sw<BITS, 2, 4>(p, sm_count, stream);
}

}  // namespace

// x, the 4-bit per-word sums, then the 8 warps' rings
size_t qmv_mixbit_smem_bytes(int bits, int64_t K, int64_t group) {
    const int64_t E = 128 / bits, sw = group >= E ? 1 : E / group;
    const MixShape sh = mix_shape(bits, K);
    const size_t ring = (size_t)sh.stages * sh.rows * 32 * (16 + (size_t)sw * 4 * (bits == 4 ? 2 : 1));
    return (((size_t)K * 4 + (bits == 4 ? (size_t)(K / 8) * 4 : 0)) + 127) / 128 * 128 + (kMixThreads / 32) * ring;
}

cudaError_t launch_qmv_mixbit(int bits, const void* qp, const void* sc, const void* bi, int G, const void* x,
                              int x_bf16, void* y, int y_bf16, int N, int K, int sm_count, cudaStream_t stream) {
    MixParams p;
    p.qp = static_cast<const uint4*>(qp);
    p.sc = static_cast<const uint16_t*>(sc);
    p.bi = static_cast<const uint16_t*>(bi);
    p.x = x;
    p.y = y;
    p.N = N;
    p.K = K;
    p.G = G;
    p.wq = (int)((int64_t)K * bits / 128);
    p.gshift = -1;
    for (int sh = 4; sh < 31; ++sh)
        if (G == (1 << sh)) p.gshift = sh;
    p.x_bf16 = x_bf16;
    p.y_bf16 = y_bf16;
    switch (bits) {
        case 2: return launch_mix_shape<2>(p, sm_count, stream);
        case 4: return launch_mix_shape<4>(p, sm_count, stream);
        case 8: return launch_mix_shape<8>(p, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dequant_mixbit(int bits, const void* qp, const void* sc, const void* bi, int G, float* out, int N,
                                  int K, int sm_count, cudaStream_t stream) {
    const unsigned grid = (unsigned)(sm_count * 8);
    const uint32_t* q = static_cast<const uint32_t*>(qp);
    const uint16_t* s = static_cast<const uint16_t*>(sc);
    const uint16_t* b = static_cast<const uint16_t*>(bi);
    switch (bits) {
        case 2: dequant_mixbit_kernel<2><<<grid, 256, 0, stream>>>(q, s, b, G, N, K, out); break;
        case 4: dequant_mixbit_kernel<4><<<grid, 256, 0, stream>>>(q, s, b, G, N, K, out); break;
        case 8: dequant_mixbit_kernel<8><<<grid, 256, 0, stream>>>(q, s, b, G, N, K, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qbw
