// Per-pixel neural shading (Pulsar Sec. 3.3: a per-pixel network turns the
// rendered feature map into RGB; Sec. 5.2: a shared per-pixel fully
// connected model conditioned on the view direction) on the 5th-generation
// tensor cores, forward and backward.
//
//   x  = [F_p (16 channels), v_p (unit view direction)]
//   h1 = ReLU(W1 x + b1), h2 = ReLU(W2 h1 + b2), y = W3 h2 + b3
//   (19 -> 64 -> 64 -> 3; matrix operands bfloat16, fp32 accumulation,
//   fp32 biases)
//
// Both kernels run persistent CTAs of 128 threads over 128-pixel tiles, one
// thread per pixel (one row of M = 128, one TMEM lane).  Per layer the
// threads write their rows of the A operand, one thread issues the layer's
// tcgen05.mma into the CTA's tensor memory and commits to an mbarrier, and
// every thread reads its accumulator row back with tcgen05.ld for the
// epilogue (ReLU and the bf16 rounding in one convert; the biases are added
// by the MMA itself, see the weight images).  The forward keeps every A
// operand in tensor memory (tcgen05.st by the threads, A-from-TMEM MMAs);
// the backward writes them to shared memory (no-swizzle K-major layout:
// 8-row x 16-byte core matrices), where its weight-gradient MMAs need them.
// Weights are packed once per call and bulk-copied by every CTA as the B
// operands (N x K, K-major).  Every mbarrier wait is bounded: on timeout the
// CTA latches an error, stops issuing and frees its tensor memory.
//
// The backward contracts over pixels for the weight gradients: the
// activation tiles the thread rows wrote (pixel x unit, K-major) are the
// same bytes as (unit x pixel) MN-major operands, so the MMA reads them in
// place and accumulates the CTA's share of dW in tensor memory across all
// its tiles; a ones column in the x and h2 tiles turns the same MMAs into
// the bias gradients.
#include "pulsar_internal.cuh"

#include <cuda_bf16.h>

namespace pulsar {
namespace {

constexpr int kRows = 128;           // pixels per tile (M = 128), one thread each
constexpr int kIn = 32;              // 19 inputs, zero padded to two K = 16 steps
constexpr int kHid = 64;
constexpr int kOutPad = 16;          // 3 outputs padded to the smallest N for M = 128

// flat parameter layout: W1 [64][19], b1 [64], W2 [64][64], b2 [64], W3 [3][64], b3 [3]
constexpr int kOffB1 = kHid * 19;
constexpr int kOffW2 = kOffB1 + kHid;
constexpr int kOffB2 = kOffW2 + kHid * kHid;
constexpr int kOffW3 = kOffB2 + kHid;
constexpr int kOffB3 = kOffW3 + 3 * kHid;
static_assert(kOffB3 + 3 == kShadeParams, "shading parameter layout");

// ------------------------------------------------------------ tcgen05 --

// Shared-memory matrix descriptor, no swizzle: start address, the byte offset
// between core matrices along K (lbo) and along M/N (sbo) -- the same roles
// for K-major and MN-major operands -- and descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// K-major unless mn_major (bits 15 and 16 mark A and B MN-major), N >> 3 at
// bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool mn_major = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (mn_major ? (3u << 15) : 0u) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(mbar))
        : "memory");
}


// 16 consecutive fp32 columns of this thread's TMEM lane (warp w owns lanes
// 32w .. 32w + 31); the values are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 16 / 32 consecutive 32-bit columns of this thread's TMEM lane; the
// stores are complete after tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::
            "r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// MMA with the A operand in tensor memory (lane = row, two bf16 per column,
// the even K element in the low half) and B in shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy shared-memory writes become visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The operands the threads wrote are complete, and every thread's earlier
// tensor-memory reads are ordered before the MMAs issued next.
__device__ __forceinline__ void operands_ready() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ __forceinline__ void tmem_alloc(uint32_t* s_taddr, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_taddr)),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
}

// Byte offset of element (row, k) in a no-swizzle K-major operand with K
// columns: core matrix (row / 8, k / 8) at (row / 8) * (K / 8) * 128 +
// (k / 8) * 128, then (row % 8) * 16 + (k % 8) * 2.
__host__ __device__ constexpr uint32_t kmajor_off(int row, int k, int K) {
    return (uint32_t)((row >> 3) * (K >> 3) * 128 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Eight consecutive K values (one 16-byte row of a core matrix) as bf16.
__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return u;
}

__device__ __forceinline__ void put8(unsigned char* tile, int row, int k, int K, const float* v) {
    *reinterpret_cast<uint4*>(tile + kmajor_off(row, k, K)) = pack8(v);
}


// The pixel's unit view direction (camera space) from its camera.
__device__ __forceinline__ void view_dir(const Frame& f, uint32_t local, float* v) {
    if (f.ortho) {
        v[0] = 0.0f;
        v[1] = 0.0f;
        v[2] = 1.0f;
        return;
    }
    const int x = (int)(local % (uint32_t)f.width), y = (int)(local / (uint32_t)f.width);
    const float a = ((float)x + 0.5f - f.cx) / f.fx, b = ((float)y + 0.5f - f.cy) / f.fy;
    const float inv = rsqrtf(a * a + b * b + 1.0f);
    v[0] = a * inv;
    v[1] = b * inv;
    v[2] = inv;
}

__device__ __forceinline__ void load_features(const float* __restrict__ features, uint64_t p,
                                              bool valid, float4 (&f)[4]) {
    const float4* fp = reinterpret_cast<const float4*>(features + p * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) f[q] = valid ? fp[q] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Layer input row: 16 features, the view direction, ones at columns 19-21,
// zeros.  The ones meet the three bf16 parts of each bias in the B operands
// (the tensor cores add the fp32 bias exactly, inside the fp32 sum), and
// column 19 turns the backward's weight-gradient contraction into the bias
// gradient.
__device__ __forceinline__ void input_row(const Frames& fs, uint32_t P1, uint64_t p, bool valid,
                                          const float4 (&f)[4], float (&in)[kIn]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        in[4 * q] = f[q].x;
        in[4 * q + 1] = f[q].y;
        in[4 * q + 2] = f[q].z;
        in[4 * q + 3] = f[q].w;
    }
#pragma unroll
    for (int k = 16; k < kIn; ++k) in[k] = (k >= 19 && k <= 21) ? 1.0f : 0.0f;
    if (valid) {
        const uint32_t cam = (uint32_t)(p / P1);
        view_dir(fs.f[cam], (uint32_t)(p - (uint64_t)cam * P1), in + 16);
    }
}

// Two fp32 values as one bf16x2 word (the first in the low half), rounded to
// nearest even; the relu form turns negative values into 0.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_relu(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// 0xFFFF in each half of a bf16x2 word of ReLU outputs that is not +-0, else
// 0: the magnitude plus 0x7FFF carries into the half's top bit exactly when
// it is non-zero, and prmt replicates that bit across the half.
__device__ __forceinline__ uint32_t nonzero_mask(uint32_t h) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(d) : "r"((h & 0x7FFF7FFFu) + 0x7FFF7FFFu));
    return d;
}

__device__ __forceinline__ void st_row16(unsigned char* tile, int row, int k, int K,
                                         const uint32_t* w) {
    *reinterpret_cast<uint4*>(tile + kmajor_off(row, k, K)) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Hidden layer epilogue: h = bf16(ReLU(D)) (D holds the bias) of this
// thread's row into columns k0 .. k0 + 63 of a K-column A operand; the bf16x2
// words stay in h for the backward's ReLU masks.  kBatch columns are read
// from tensor memory per wait (registers against latency).
template <int kBatch>
__device__ __forceinline__ void relu_row(uint32_t taddr, unsigned char* tile, int row, int K,
                                         int k0, uint32_t (&h)[kHid / 2]) {
#pragma unroll
    for (int c0 = 0; c0 < kHid; c0 += kBatch) {
        uint32_t r[kBatch / 16][16];
#pragma unroll
        for (int q = 0; q < kBatch / 16; ++q) tmem_ld16(taddr + (uint32_t)(c0 + 16 * q), r[q]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kBatch / 2; ++j)
            h[c0 / 2 + j] = bf16x2_relu(__uint_as_float(r[j / 8][(2 * j) % 16]),
                                        __uint_as_float(r[j / 8][(2 * j + 1) % 16]));
#pragma unroll
        for (int q = 0; q < kBatch / 8; ++q)
            st_row16(tile, row, k0 + c0 + 8 * q, K, h + c0 / 2 + 4 * q);
    }
}

// Backward epilogue: Q(D * [h > 0]) of this thread's row into columns
// k0 .. k0 + 63 (h: the layer's ReLU output words), all 64 columns per wait.
__device__ __forceinline__ void masked_row(uint32_t taddr, const uint32_t (&h)[kHid / 2],
                                           unsigned char* tile, int row, int K, int k0) {
    uint32_t r[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q) tmem_ld16(taddr + (uint32_t)(16 * q), r[q]);
    tmem_wait_ld();
    uint32_t g[kHid / 2];
#pragma unroll
    for (int j = 0; j < kHid / 2; ++j)
        g[j] = bf16x2(__uint_as_float(r[j / 8][(2 * j) % 16]),
                      __uint_as_float(r[j / 8][(2 * j + 1) % 16])) &
               nonzero_mask(h[j]);
#pragma unroll
    for (int q = 0; q < kHid / 8; ++q) st_row16(tile, row, k0 + 8 * q, K, g + 4 * q);
}

// Both epilogues of the backward's second round from one wait: h2 =
// bf16(ReLU(z2)) into the h2 tile, then Q(g2 * [h2 > 0]) into the g tile.
__device__ __forceinline__ void relu_and_masked_row(uint32_t tz, uint32_t tg, unsigned char* htile,
                                                    int hK, unsigned char* gtile, int gK, int gk0,
                                                    int row) {
    uint32_t z[4][16], g[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        tmem_ld16(tz + (uint32_t)(16 * q), z[q]);
        tmem_ld16(tg + (uint32_t)(16 * q), g[q]);
    }
    tmem_wait_ld();
    uint32_t h[kHid / 2], w[kHid / 2];
#pragma unroll
    for (int j = 0; j < kHid / 2; ++j) {
        h[j] = bf16x2_relu(__uint_as_float(z[j / 8][(2 * j) % 16]),
                           __uint_as_float(z[j / 8][(2 * j + 1) % 16]));
        w[j] = bf16x2(__uint_as_float(g[j / 8][(2 * j) % 16]),
                      __uint_as_float(g[j / 8][(2 * j + 1) % 16])) &
               nonzero_mask(h[j]);
    }
#pragma unroll
    for (int q = 0; q < kHid / 8; ++q) {
        st_row16(htile, row, 8 * q, hK, h + 4 * q);
        st_row16(gtile, row, gk0 + 8 * q, gK, w + 4 * q);
    }
}

// Step `bytes` into the operand a descriptor describes (the address field
// counts 16-byte units; shared addresses stay far below its 2^18-byte range).
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// One K-major MMA chain: D = sum over `steps` K = 16 steps of A_s B_s^T, A
// and B advancing 256 bytes (two core matrices) per step.
__device__ __forceinline__ void mma_chain(uint32_t d, uint64_t a, uint64_t b, int steps,
                                          uint32_t idesc, uint32_t acc0) {
    for (int s = 0; s < steps; ++s)
        mma_bf16(d, desc_at(a, 256u * s), desc_at(b, 256u * s), idesc, s > 0 ? 1u : acc0);
}

// ================================================================ weights --
// The weights as the kernels hold them in shared memory: bf16 B operands
// (N x K, K-major, zero padded), one image per kernel, written once per call
// and bulk-copied by every CTA.  Each fp32 bias b is split exactly into three
// bf16 parts (b = hi + mid + lo: 8 + 8 + 8 significant bits) placed where the
// A operand holds ones: columns 19-21 of layer 1's x, and for layers 2 and 3
// an extra K step over x's columns 16-31 (view direction, ones, zeros) in
// front of the hidden units.
constexpr int kKB = 16 + kHid;   // layers 2, 3: the bias K step, then the 64 units

struct FwdImage {   // W1 | b1 [64 x 32], b2 | W2 [64 x 80], b3 | W3 [16 x 80]
    static constexpr int w1 = 0;
    static constexpr int w2 = w1 + kHid * kIn * 2;
    static constexpr int w3 = w2 + kHid * kKB * 2;
    static constexpr int bytes = w3 + kOutPad * kKB * 2;
};
struct BwdImage {   // W1 | b1, b2 | W2, W3^T [64 x 16], W2^T [64 x 64], W1^T [16 x 64]
    static constexpr int w1 = 0;
    static constexpr int w2 = w1 + kHid * kIn * 2;
    static constexpr int w3t = w2 + kHid * kKB * 2;
    static constexpr int w2t = w3t + kHid * 16 * 2;
    static constexpr int w1t = w2t + kHid * kHid * 2;
    static constexpr int bytes = w1t + 16 * kHid * 2;
};
static_assert(FwdImage::bytes % 16 == 0 && BwdImage::bytes % 16 == 0, "bulk copy sizes");
constexpr int kImageBytes = FwdImage::bytes + BwdImage::bytes;

// Part i (0 hi, 1 mid, 2 lo) of the exact three-way bf16 split of b (each
// remainder is exact in fp32).
__device__ __forceinline__ float bias_part(float b, int i) {
    const float hi = __bfloat162float(__float2bfloat16_rn(b));
    if (i == 0) return hi;
    const float r = b - hi;
    const float mid = __bfloat162float(__float2bfloat16_rn(r));
    return i == 1 ? mid : r - mid;
}

enum Operand { kW1b, kW2b, kW3b, kW3t, kW2t, kW1t };

// Element (n, k) of a B operand.
__device__ float operand_value(Operand o, int n, int k, const float* __restrict__ prm) {
    const float* W1 = prm;
    const float* W2 = prm + kOffW2;
    const float* W3 = prm + kOffW3;
    switch (o) {
        case kW1b:   // [64 x 32]: W1 (19), the parts of b1, zeros
            return k < 19 ? W1[n * 19 + k] : (k <= 21 ? bias_part(prm[kOffB1 + n], k - 19) : 0.0f);
        case kW2b:   // [64 x 80]: parts of b2 at 3-5 of the bias step, then W2
            return k >= 16 ? W2[n * kHid + k - 16]
                           : (k >= 3 && k <= 5 ? bias_part(prm[kOffB2 + n], k - 3) : 0.0f);
        case kW3b:   // [16 x 80]: rows 0-2 as kW2b with b3 and W3
            if (n >= 3) return 0.0f;
            return k >= 16 ? W3[n * kHid + k - 16]
                           : (k >= 3 && k <= 5 ? bias_part(prm[kOffB3 + n], k - 3) : 0.0f);
        case kW3t: return k < 3 ? W3[k * kHid + n] : 0.0f;   // [64 x 16]
        case kW2t: return W2[k * kHid + n];                   // [64 x 64]
        default:   return W1[k * 19 + n];                     // [16 x 64] kW1t
    }
}

struct PackSeg {
    int offset, rows, K;
    Operand o;
};
__device__ constexpr PackSeg kPack[] = {
    {FwdImage::w1, kHid, kIn, kW1b},
    {FwdImage::w2, kHid, kKB, kW2b},
    {FwdImage::w3, kOutPad, kKB, kW3b},
    {FwdImage::bytes + BwdImage::w1, kHid, kIn, kW1b},
    {FwdImage::bytes + BwdImage::w2, kHid, kKB, kW2b},
    {FwdImage::bytes + BwdImage::w3t, kHid, 16, kW3t},
    {FwdImage::bytes + BwdImage::w2t, kHid, kHid, kW2t},
    {FwdImage::bytes + BwdImage::w1t, 16, kHid, kW1t},
};
constexpr int kPackElems = kHid * kIn * 2 + kHid * kKB * 2 + kOutPad * kKB + kHid * 16 +
                           kHid * kHid + 16 * kHid;

__global__ void k_shade_pack(const float* __restrict__ params, unsigned char* __restrict__ img) {
    pdl_begin();
    int e = blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll
    for (int s = 0; s < (int)(sizeof(kPack) / sizeof(kPack[0])); ++s) {
        const PackSeg g = kPack[s];
        if (e < g.rows * g.K) {
            const int n = e / g.K, k = e % g.K;
            reinterpret_cast<__nv_bfloat16*>(img + g.offset)[kmajor_off(n, k, g.K) / 2] =
                __float2bfloat16_rn(operand_value(g.o, n, k, params));
            return;
        }
        e -= g.rows * g.K;
    }
}

// ================================================================ forward --
// Every A operand lives in tensor memory, written by the threads with
// tcgen05.st (two bf16 per 32-bit column, the pixel's row = its lane), so
// shared memory holds only the weights and no operand passes through it.
// Columns: the accumulator 0-63 (every layer), x 64-79 (32 inputs; its
// columns 72-79 -- view direction, ones -- are the bias step of layers 2
// and 3), the hidden units 80-111.
constexpr int kFwdCols = 128;
constexpr uint32_t kColX = 64, kColH = 80;
constexpr int kXH = kIn + kHid;   // backward A tile columns: x (32), then h1 (64)

struct FwdSmem {
    static constexpr int img = 0;                         // FwdImage
    static constexpr int w1 = img + FwdImage::w1;
    static constexpr int w2 = img + FwdImage::w2;
    static constexpr int w3 = img + FwdImage::w3;
    static constexpr int mbar = img + FwdImage::bytes;    // u64: MMA completion
    static constexpr int wbar = mbar + 8;                 // u64: weights landed
    static constexpr int taddr = wbar + 8;                // u32
    static constexpr int bytes = taddr + 8;
};

// The threads' tensor-memory stores are complete, and every thread's earlier
// tensor-memory accesses are ordered before the MMAs issued next.
__device__ __forceinline__ void tmem_operands_ready() {
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__global__ void __launch_bounds__(kRows)
k_shade_forward(Frames fs, Workspace w, const float* __restrict__ features,
                const unsigned char* __restrict__ img, float* __restrict__ rgb) {
    pdl_begin();
    using L = FwdSmem;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::mbar);
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + L::wbar);
    uint32_t* s_taddr = reinterpret_cast<uint32_t*>(smem + L::taddr);
    const int tid = threadIdx.x, warp = tid >> 5;
    const Frame& f0 = fs.f[0];
    const uint64_t n_pix = f0.pix_all;
    const uint32_t P1 = (uint32_t)(f0.width * f0.height);
    const uint32_t n_tiles = (uint32_t)((n_pix + kRows - 1) / kRows);
    const uint64_t stride = (uint64_t)gridDim.x * kRows;

    if (tid == 0) {
        mbar_init(mbar);
        mbar_init(wbar);
        fence_async_smem();
        bulk_load(smem + L::img, img, FwdImage::bytes, wbar);
    }
    if (warp == 0) tmem_alloc(s_taddr, kFwdCols);
    operands_ready();
    const uint32_t tmem = *s_taddr;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's TMEM lanes
    // B descriptors (K-major; core matrices 128 B apart along K, a row block apart along N)
    const uint64_t d_w1 = smem_desc(smem_u32(smem + L::w1), 128, (kIn / 8) * 128);
    const uint64_t d_w2 = smem_desc(smem_u32(smem + L::w2), 128, (kKB / 8) * 128);
    const uint64_t d_w3 = smem_desc(smem_u32(smem + L::w3), 128, (kKB / 8) * 128);
    uint32_t phase = 0;
    bool ok = true;

    // test hook: issue nothing, so the first wait runs out
    const bool issue = (w.state->inject & kInjectShadeTimeout) == 0u;
    uint64_t p = (uint64_t)blockIdx.x * kRows + tid;
    float4 fcur[4];
    load_features(features, p, p < n_pix, fcur);
    ok = __syncthreads_and(mbar_wait(wbar, 0));   // the weights are in
    for (uint32_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, p += stride) {
        const bool valid = p < n_pix;
        {
            float in[kIn];
            input_row(fs, P1, p, valid, fcur, in);
            uint32_t xw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) xw[j] = bf16x2(in[2 * j], in[2 * j + 1]);
            tmem_st16(trow + kColX, xw);
        }
        // the next tile's features load while this tile runs through the tensor cores
        load_features(features, p + stride, p + stride < n_pix, fcur);
        tmem_operands_ready();
        if (tid == 0 && issue) {
#pragma unroll
            for (int s2 = 0; s2 < kIn / 16; ++s2)
                mma_bf16_ta(tmem, tmem + kColX + 8 * s2, desc_at(d_w1, 256u * s2),
                            idesc_bf16(kRows, kHid), s2 > 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));   // one decision for all
        ++phase;
        tc_fence_after();
        if (!ok) break;
#pragma unroll
        for (int layer = 2; layer <= 3; ++layer) {
            {   // h = bf16(ReLU(D)) of this row into the hidden columns
                uint32_t r[4][16], h[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(trow + (uint32_t)(16 * q), r[q]);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    h[j] = bf16x2_relu(__uint_as_float(r[j / 8][(2 * j) % 16]),
                                       __uint_as_float(r[j / 8][(2 * j + 1) % 16]));
                tmem_st32(trow + kColH, h);
            }
            tmem_operands_ready();
            if (tid == 0) {   // the bias step over x's columns 16-31, then the 64 hidden units
                const uint64_t d_w = layer == 2 ? d_w2 : d_w3;
                const uint32_t id = idesc_bf16(kRows, layer == 2 ? kHid : kOutPad);
                mma_bf16_ta(tmem, tmem + kColX + 8, d_w, id, 0);
#pragma unroll
                for (int s2 = 0; s2 < kHid / 16; ++s2)
                    mma_bf16_ta(tmem, tmem + kColH + 8 * s2, desc_at(d_w, 256u * (s2 + 1)), id, 1);
                mma_commit(mbar);
            }
            ok = __syncthreads_and(mbar_wait(mbar, phase & 1));
            ++phase;
            tc_fence_after();
            if (!ok) break;
        }
        if (!ok) break;
        // y = D3; the next tile's stores need no further barrier: layer 3 is
        // complete and this row's accumulator is read here
        uint32_t r[16];
        tmem_ld16(trow, r);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
            for (int o = 0; o < 3; ++o) rgb[p * 3 + o] = __uint_as_float(r[o]);
        }
    }
    if (!ok) {
        // a copy or an MMA did not complete in time: report it, give both
        // one more bounded wait, then release the tensor memory regardless
        if (tid == 0) atomicOr(&w.state->error, kErrTimeout);
        mbar_wait(wbar, 0);
        if (phase > 0) mbar_wait(mbar, (phase - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kFwdCols);
}

// =============================================================== backward --
// Gradients of L = sum_p <dY_p, y_p>, straight through the bf16 roundings:
//   g2 = (W3^T Q(dY)) * [z2 > 0],  g1 = (W2^T Q(g2)) * [z1 > 0],  dF = (W1^T Q(g1))[:16]
//   rows 0..63 / 64..127 of  sum_p [Q(g1) ; Q(g2)] [Q(x), 1 | Q(h1)]^T  hold
//     [dW1 | db1 | .] and [. | db2 | dW2]
//   rows 0..63 / 64 of  sum_p [Q(h2) ; 1] Q(dY)^T  hold dW3^T and db3^T
// ([z > 0] is read as [Q(ReLU(z)) != 0]: they differ only for 0 < z below
// the smallest bfloat16, far inside the fp32 error of z.)
constexpr int kBwdCols = 256;
constexpr int kGG = 128;    // Q(g1) (64), Q(g2) (64)
constexpr int kH2 = 72;     // Q(h2) (64), 1, zero pad
constexpr int kDY = 16;     // Q(dY) (3), zero pad
constexpr uint32_t kColZ1 = 0, kColZ2 = 64, kColG2 = 0, kColG1 = 64, kColDX = 0;
constexpr uint32_t kColAccXH = 128;   // 96 columns
constexpr uint32_t kColAccY = 224;    // 16 columns

struct BwdSmem {
    static constexpr int xh = 0;                            // [128 x 96]: x | h1
    static constexpr int gg = xh + kRows * kXH * 2;         // [128 x 128]
    static constexpr int h2 = gg + kRows * kGG * 2;         // [128 x 72]
    static constexpr int dy = h2 + kRows * kH2 * 2;         // [128 x 16]
    static constexpr int img = dy + kRows * kDY * 2;        // BwdImage
    static constexpr int w1 = img + BwdImage::w1;
    static constexpr int w2 = img + BwdImage::w2;
    static constexpr int w3t = img + BwdImage::w3t;
    static constexpr int w2t = img + BwdImage::w2t;
    static constexpr int w1t = img + BwdImage::w1t;
    static constexpr int mbar = img + BwdImage::bytes;      // u64: the dF chain's MMAs
    static constexpr int gbar = mbar + 8;                   // u64: the weight-gradient MMAs
    static constexpr int wbar = gbar + 8;                   // u64: weights landed
    static constexpr int taddr = wbar + 8;
    static constexpr int bytes = taddr + 8;
};
// Read MN-major, the [Q(h2) | 1] tile spans 16 groups of 8 units per pixel
// group of which it holds 9: the last instruction's reads end 19328 bytes
// from its start, inside the dy tile that follows.
static_assert(BwdSmem::dy + kRows * kDY * 2 - BwdSmem::h2 >=
                  7 * (2 * kH2 * 16) + 15 * 128 + kH2 * 16 + 128,
              "MN-major read of the h2 tile stays inside shared memory");

__global__ void __launch_bounds__(kRows, 2)
k_shade_backward(Frames fs, Workspace w, const float* __restrict__ features,
                 const unsigned char* __restrict__ img, const float* __restrict__ grad_rgb,
                 float* __restrict__ grad_features, float* __restrict__ part) {
    pdl_begin();
    using L = BwdSmem;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::mbar);
    uint64_t* gbar = reinterpret_cast<uint64_t*>(smem + L::gbar);
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + L::wbar);
    uint32_t* s_taddr = reinterpret_cast<uint32_t*>(smem + L::taddr);
    const int tid = threadIdx.x, warp = tid >> 5;
    const Frame& f0 = fs.f[0];
    const uint64_t n_pix = f0.pix_all;
    const uint32_t P1 = (uint32_t)(f0.width * f0.height);
    const uint32_t n_tiles = (uint32_t)((n_pix + kRows - 1) / kRows);
    const uint64_t stride = (uint64_t)gridDim.x * kRows;

    {   // the constant [1, 0, ...] group of the h2 tile
        const float one[8] = {1.0f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        put8(smem + L::h2, tid, kHid, kH2, one);
    }
    if (tid == 0) {
        mbar_init(mbar);
        mbar_init(gbar);
        mbar_init(wbar);
        fence_async_smem();
        bulk_load(smem + L::img, img, BwdImage::bytes, wbar);
    }
    if (warp == 0) tmem_alloc(s_taddr, kBwdCols);
    operands_ready();
    const uint32_t tmem = *s_taddr;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    const uint32_t sxh = smem_u32(smem + L::xh), sgg = smem_u32(smem + L::gg),
                   sh2 = smem_u32(smem + L::h2), sdy = smem_u32(smem + L::dy);
    // K-major descriptors: core matrices 128 B apart along K, a row block apart along M/N
    const uint64_t d_xh = smem_desc(sxh, 128, (kXH / 8) * 128);
    const uint64_t d_gg = smem_desc(sgg, 128, (kGG / 8) * 128);
    const uint64_t d_dy = smem_desc(sdy, 128, (kDY / 8) * 128);
    const uint64_t d_w1 = smem_desc(smem_u32(smem + L::w1), 128, (kIn / 8) * 128);
    const uint64_t d_w2 = smem_desc(smem_u32(smem + L::w2), 128, (kKB / 8) * 128);
    const uint64_t d_w3t = smem_desc(smem_u32(smem + L::w3t), 128, (kDY / 8) * 128);
    const uint64_t d_w2t = smem_desc(smem_u32(smem + L::w2t), 128, (kHid / 8) * 128);
    const uint64_t d_w1t = smem_desc(smem_u32(smem + L::w1t), 128, (kHid / 8) * 128);
    // MN-major descriptors of the pixel contractions: groups of 8 units 128 B
    // apart (M/N), groups of 8 pixels one row block apart (K); 16 pixels per
    // instruction = two row blocks
    const uint64_t m_gg = smem_desc(sgg, (kGG / 8) * 128, 128);
    const uint64_t m_xh = smem_desc(sxh, (kXH / 8) * 128, 128);
    const uint64_t m_h2 = smem_desc(sh2, (kH2 / 8) * 128, 128);
    const uint64_t m_dy = smem_desc(sdy, (kDY / 8) * 128, 128);
    uint32_t phase = 0, gphase = 0;
    bool ok = true;
    uint32_t acc = 0;   // 0 until the first tile's weight-gradient MMAs are issued
    uint32_t h1[kHid / 2];

    // test hook: issue nothing, so the first wait runs out
    const bool issue = (w.state->inject & kInjectShadeTimeout) == 0u;
    uint64_t p = (uint64_t)blockIdx.x * kRows + tid;
    float4 fcur[4];
    float dcur[3];
    load_features(features, p, p < n_pix, fcur);
#pragma unroll
    for (int o = 0; o < 3; ++o) dcur[o] = p < n_pix ? grad_rgb[p * 3 + o] : 0.0f;
    ok = __syncthreads_and(mbar_wait(wbar, 0));   // the weights are in
    for (uint32_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, p += stride) {
        const bool valid = p < n_pix;
        if (acc) {   // the previous tile's weight-gradient MMAs still read x, h1, g, dy
            ok = __syncthreads_and(mbar_wait(gbar, gphase & 1));
            ++gphase;
            if (!ok) break;
        }
        {
            float in[kIn];
            input_row(fs, P1, p, valid, fcur, in);
#pragma unroll
            for (int j = 0; j < kIn / 8; ++j) put8(smem + L::xh, tid, 8 * j, kXH, in + 8 * j);
            const uint32_t d[8] = {bf16x2(dcur[0], dcur[1]), bf16x2(dcur[2], 0.0f), 0u, 0u,
                                   0u, 0u, 0u, 0u};
            st_row16(smem + L::dy, tid, 0, kDY, d);
            st_row16(smem + L::dy, tid, 8, kDY, d + 4);
        }
        {   // the next tile's inputs load while this tile runs through the tensor cores
            const uint64_t pn = p + stride;
            const bool vn = pn < n_pix;
            load_features(features, pn, vn, fcur);
#pragma unroll
            for (int o = 0; o < 3; ++o) dcur[o] = vn ? grad_rgb[pn * 3 + o] : 0.0f;
        }
        operands_ready();
        // ---- round 1: z1 = W1 Q(x) + b1
        if (tid == 0 && issue) {
            mma_chain(tmem + kColZ1, d_xh, d_w1, kIn / 16, idesc_bf16(kRows, kHid), 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        relu_row<64>(trow + kColZ1, smem + L::xh, tid, kXH, kIn, h1);
        operands_ready();
        // ---- round 2: z2 = W2 Q(h1) + b2 (bias step over x's columns 16-31), and W3^T Q(dY)
        if (tid == 0) {
            mma_chain(tmem + kColZ2, desc_at(d_xh, 256), d_w2, kKB / 16, idesc_bf16(kRows, kHid), 0);
            mma_bf16(tmem + kColG2, d_dy, d_w3t, idesc_bf16(kRows, kHid), 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        relu_and_masked_row(trow + kColZ2, trow + kColG2, smem + L::h2, kH2, smem + L::gg, kGG,
                            kHid, tid);   // h2, Q(g2)
        operands_ready();
        // ---- round 3: W2^T Q(g2) (committed alone); then accumulate
        // [Q(h2) ; 1] Q(dY)^T over the tile's pixels behind it
        if (tid == 0) {
            mma_chain(tmem + kColG1, desc_at(d_gg, kHid / 8 * 128), d_w2t, kHid / 16,
                      idesc_bf16(kRows, kHid), 0);
            mma_commit(mbar);
            for (int q = 0; q < kRows; q += 16)
                mma_bf16(tmem + kColAccY, desc_at(m_h2, (q / 8) * (kH2 / 8) * 128),
                         desc_at(m_dy, (q / 8) * (kDY / 8) * 128), idesc_bf16(kRows, kDY, true),
                         acc | (uint32_t)(q > 0));
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        masked_row(trow + kColG1, h1, smem + L::gg, tid, kGG, 0);   // Q(g1)
        operands_ready();
        // ---- round 4: dF = (W1^T Q(g1))[:16] (committed alone); then accumulate
        // [Q(g1) ; Q(g2)] [Q(x), 1 | Q(h1)]^T behind it, on its own barrier
        if (tid == 0) {
            mma_chain(tmem + kColDX, d_gg, d_w1t, kHid / 16, idesc_bf16(kRows, 16), 0);
            mma_commit(mbar);
            for (int q = 0; q < kRows; q += 16)
                mma_bf16(tmem + kColAccXH, desc_at(m_gg, (q / 8) * (kGG / 8) * 128),
                         desc_at(m_xh, (q / 8) * (kXH / 8) * 128), idesc_bf16(kRows, kXH, true),
                         acc | (uint32_t)(q > 0));
            mma_commit(gbar);
        }
        acc = 1;
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        {
            uint32_t r[16];
            tmem_ld16(trow + kColDX, r);
            tmem_wait_ld();
            if (valid && grad_features) {
                float4* gf = reinterpret_cast<float4*>(grad_features + p * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    gf[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                        __uint_as_float(r[4 * q + 2]),
                                        __uint_as_float(r[4 * q + 3]));
            }
        }
    }
    if (ok && acc) {   // the last tile's weight-gradient MMAs
        ok = __syncthreads_and(mbar_wait(gbar, gphase & 1));
        ++gphase;
        tc_fence_after();
    }
    // ---- this CTA's share of the weight gradients: TMEM lane = output row
    float* mine = part + (size_t)blockIdx.x * kShadeParams;
    if (ok) {
        const int m = tid & (kHid - 1);
        const bool lower = tid < kHid;   // rows of Q(g1), else of Q(g2)
#pragma unroll 1
        for (int c0 = 0; c0 < kXH; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(trow + kColAccXH + (uint32_t)c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                const float v = __uint_as_float(r[j]);
                if (col < 19 && lower) mine[m * 19 + col] = v;
                if (col == 19) mine[(lower ? kOffB1 : kOffB2) + m] = v;
                if (col >= kIn && !lower) mine[kOffW2 + m * kHid + (col - kIn)] = v;
            }
        }
        uint32_t r[16];
        tmem_ld16(trow + kColAccY, r);
        tmem_wait_ld();
#pragma unroll
        for (int o = 0; o < 3; ++o) {
            if (lower) mine[kOffW3 + o * kHid + m] = __uint_as_float(r[o]);
            if (tid == kHid) mine[kOffB3 + o] = __uint_as_float(r[o]);
        }
    } else {
        // a copy or an MMA did not complete in time: report it, give each
        // barrier one more bounded wait, then release the tensor memory
        if (tid == 0) atomicOr(&w.state->error, kErrTimeout);
        mbar_wait(wbar, 0);
        if (phase > 0) mbar_wait(mbar, (phase - 1) & 1);
        if (acc) mbar_wait(gbar, gphase & 1);
        for (int e = tid; e < kShadeParams; e += kRows) mine[e] = 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kBwdCols);
}

// Sum of the CTAs' weight-gradient shares in a fixed order, in float-pair
// arithmetic (Knuth's TwoSum per addition, ~2^-44 relative: the accuracy of
// an fp64 sum of these few hundred terms at fp32 speed, where this part's
// fp64 rate is a small fraction of it): a block takes 32 parameters; warp w
// sums the shares w, w + 16, ... with four independent accumulators (loads in
// flight), the warps combine in order.
constexpr int kReduceWarps = 16;

__global__ void __launch_bounds__(32 * kReduceWarps)
k_shade_reduce(const float* __restrict__ part, int n_part, float* __restrict__ grad_params) {
    pdl_begin();
    __shared__ float2 acc[kReduceWarps][32];
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + lane;
    FPair s[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
    if (i < kShadeParams) {
        int c = wp;
        for (; c + 3 * kReduceWarps < n_part; c += 4 * kReduceWarps) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = part[(size_t)(c + u * kReduceWarps) * kShadeParams + i];
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] = pp_add(s[u], FPair{v[u], 0.0f});
        }
        for (; c < n_part; c += kReduceWarps)
            s[0] = pp_add(s[0], FPair{part[(size_t)c * kShadeParams + i], 0.0f});
    }
    const FPair t4 = pp_add(pp_add(s[0], s[1]), pp_add(s[2], s[3]));
    acc[wp][lane] = make_float2(t4.hi, t4.lo);
    __syncthreads();
    if (wp == 0 && i < kShadeParams) {
        FPair t = {0.0f, 0.0f};
#pragma unroll
        for (int w2 = 0; w2 < kReduceWarps; ++w2) t = pp_add(t, FPair{acc[w2][lane].x, acc[w2][lane].y});
        grad_params[i] = __fadd_rn(t.hi, t.lo);
    }
}

// CTAs of a kernel resident per SM, from the documented limits: shared
// memory (with the per-block reserve), registers, resident blocks, and no
// more than the tensor memory (512 columns) holds.
int resident(const void* kernel, int bytes, int tmem_cols) {
    int dev = 0;
    cudaFuncAttributes fa;
    cudaDeviceProp pr;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
        cudaGetDeviceProperties(&pr, dev) != cudaSuccess)
        return 0;
    const size_t per_block = (size_t)bytes + fa.sharedSizeBytes + pr.reservedSharedMemPerBlock;
    int n = (int)(pr.sharedMemPerMultiprocessor / per_block);
    const int regs = fa.numRegs * kRows;
    if (regs > 0 && pr.regsPerMultiprocessor / regs < n) n = pr.regsPerMultiprocessor / regs;
    if (pr.maxBlocksPerMultiProcessor < n) n = pr.maxBlocksPerMultiProcessor;
    if (512 / tmem_cols < n) n = 512 / tmem_cols;
    return n;
}

}  // namespace

size_t shade_image_bytes() { return kImageBytes; }

cudaError_t prepare_shade(ShadeLaunch* sl) {
    cudaError_t e = cudaFuncSetAttribute(k_shade_forward,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, FwdSmem::bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_shade_backward, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BwdSmem::bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_shade_forward, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 100);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_shade_backward, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 100);
    if (e != cudaSuccess) return e;
    sl->fwd_per_sm = resident((const void*)k_shade_forward, FwdSmem::bytes, kFwdCols);
    sl->bwd_per_sm = resident((const void*)k_shade_backward, BwdSmem::bytes, kBwdCols);
    return sl->fwd_per_sm > 0 && sl->bwd_per_sm > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t launch_shade_forward(const Frames& fs, const Workspace& w, const float* features,
                                 const float* params, float* rgb, int grid_cap,
                                 cudaStream_t stream) {
    const uint64_t n_tiles = (fs.f[0].pix_all + kRows - 1) / kRows;
    if (n_tiles == 0) return cudaSuccess;
    const int grid = (int)(n_tiles < (uint64_t)grid_cap ? n_tiles : (uint64_t)grid_cap);
    cudaError_t e = launch_pdl(k_shade_pack, dim3((kPackElems + 255) / 256), dim3(256), 0, stream,
                               params, w.shade_img);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_shade_forward, dim3(grid), dim3(kRows), FwdSmem::bytes, stream, fs, w,
                      features, (const unsigned char*)w.shade_img, rgb);
}

cudaError_t launch_shade_backward(const Frames& fs, const Workspace& w, const float* features,
                                  const float* params, const float* grad_rgb,
                                  float* grad_features, float* grad_params, int grid_cap,
                                  cudaStream_t stream) {
    const uint64_t n_tiles = (fs.f[0].pix_all + kRows - 1) / kRows;
    if (n_tiles == 0)
        return cudaMemsetAsync(grad_params, 0, kShadeParams * sizeof(float), stream);
    const int grid = (int)(n_tiles < (uint64_t)grid_cap ? n_tiles : (uint64_t)grid_cap);
    cudaError_t e = launch_pdl(k_shade_pack, dim3((kPackElems + 255) / 256), dim3(256), 0, stream,
                               params, w.shade_img);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_shade_backward, dim3(grid), dim3(kRows), BwdSmem::bytes, stream, fs, w,
                   features, (const unsigned char*)(w.shade_img + FwdImage::bytes), grad_rgb,
                   grad_features, w.shade_part);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_shade_reduce, dim3((kShadeParams + 31) / 32), dim3(32 * kReduceWarps), 0,
                      stream, (const float*)w.shade_part, grid, grad_params);
}

}  // namespace pulsar
