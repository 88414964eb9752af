// Per-pixel neural shading (Pulsar Sec. 3.3: a per-pixel network turns the
// rendered feature map into RGB; Sec. 5.2: a shared per-pixel fully
// connected model conditioned on the view direction) on the 5th-generation
// tensor cores.
//
//   x  = [F_p (16 channels), v_p (unit view direction)]
//   h1 = ReLU(W1 x + b1), h2 = ReLU(W2 h1 + b2), y = W3 h2 + b3
//   (19 -> 64 -> 64 -> 3; matrix operands bfloat16, fp32 accumulation,
//   fp32 biases)
//
// k_shade_forward  persistent CTAs of 128 threads, one 128-pixel tile at a
//     time, one thread per pixel: the thread writes its pixel's bf16 inputs
//     into the tile's A operand in shared memory (no-swizzle K-major layout:
//     8-row x 16-byte core matrices, 128 B apart along K), one thread issues
//     the layer's tcgen05.mma (M = 128, K = 16 per instruction) into the
//     CTA's tensor memory and commits to an mbarrier, and every thread reads
//     its row back with tcgen05.ld, adds the bias, applies the ReLU and
//     writes the next layer's A operand.  Weights are staged once per CTA as
//     the B operands (N x K, K-major).  Every mbarrier wait is bounded: on
//     timeout the CTA latches an error, stops issuing and frees its tensor
//     memory.
#include "pulsar_internal.cuh"

#include <cuda_bf16.h>

namespace pulsar {
namespace {

constexpr int kShadeThreads = 128;   // one thread per pixel of a tile (M = 128)
constexpr int kIn = 32;              // 19 inputs, zero padded to two K = 16 steps
constexpr int kHid = 64;
constexpr int kOutPad = 16;          // 3 outputs padded to the smallest N for M = 128
constexpr int kTmemCols = 128;       // D1 / D3 in columns 0.., D2 in 64..
constexpr uint32_t kWaitLimit = 1u << 24;

// ------------------------------------------------------------ tcgen05 --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor, no swizzle: start address, the byte offset
// of the next core matrix along K (lbo) and along M/N (sbo), descriptor
// version 1 (bit 46).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
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

// Bounded wait for the mbarrier phase of the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(mbar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp w owns lanes
// 32w .. 32w + 31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
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

struct ShadeSmem {
    static constexpr int w1 = 0;                                   // B [64 x 32]
    static constexpr int w2 = w1 + kHid * kIn * 2;                 // B [64 x 64]
    static constexpr int w3 = w2 + kHid * kHid * 2;                // B [16 x 64]
    static constexpr int x = w3 + kOutPad * kHid * 2;              // A [128 x 32]
    static constexpr int h1 = x + kShadeThreads * kIn * 2;         // A [128 x 64]
    static constexpr int h2 = h1 + kShadeThreads * kHid * 2;       // A [128 x 64]
    static constexpr int bias = h2 + kShadeThreads * kHid * 2;     // fp32 b1[64] b2[64] b3[16]
    static constexpr int mbar = bias + (2 * kHid + kOutPad) * 4;   // u64
    static constexpr int taddr = mbar + 8;                         // u32
    static constexpr int bytes = taddr + 8;
};

// Stage the weights as B operands (N x K, K-major, zero padded) and the biases.
__device__ void stage_weights(unsigned char* smem, const float* __restrict__ params) {
    using L = ShadeSmem;
    const float* W1 = params;                        // [64][19]
    const float* b1 = W1 + kHid * 19;
    const float* W2 = b1 + kHid;                     // [64][64]
    const float* b2 = W2 + kHid * kHid;
    const float* W3 = b2 + kHid;                     // [3][64]
    const float* b3 = W3 + 3 * kHid;
    __nv_bfloat16* s1 = reinterpret_cast<__nv_bfloat16*>(smem + L::w1);
    __nv_bfloat16* s2 = reinterpret_cast<__nv_bfloat16*>(smem + L::w2);
    __nv_bfloat16* s3 = reinterpret_cast<__nv_bfloat16*>(smem + L::w3);
    for (int e = threadIdx.x; e < kHid * kIn; e += blockDim.x) {
        const int n = e / kIn, k = e % kIn;
        s1[kmajor_off(n, k, kIn) / 2] = __float2bfloat16_rn(k < 19 ? W1[n * 19 + k] : 0.0f);
    }
    for (int e = threadIdx.x; e < kHid * kHid; e += blockDim.x) {
        const int n = e / kHid, k = e % kHid;
        s2[kmajor_off(n, k, kHid) / 2] = __float2bfloat16_rn(W2[n * kHid + k]);
    }
    for (int e = threadIdx.x; e < kOutPad * kHid; e += blockDim.x) {
        const int n = e / kHid, k = e % kHid;
        s3[kmajor_off(n, k, kHid) / 2] = __float2bfloat16_rn(n < 3 ? W3[n * kHid + k] : 0.0f);
    }
    float* sb = reinterpret_cast<float*>(smem + L::bias);
    for (int e = threadIdx.x; e < 2 * kHid + kOutPad; e += blockDim.x)
        sb[e] = e < kHid ? b1[e] : (e < 2 * kHid ? b2[e - kHid] : (e - 2 * kHid < 3 ? b3[e - 2 * kHid] : 0.0f));
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

__global__ void __launch_bounds__(kShadeThreads)
k_shade_forward(Frames fs, Workspace w, const float* __restrict__ features,
                const float* __restrict__ params, float* __restrict__ rgb) {
    using L = ShadeSmem;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::mbar);
    uint32_t* s_taddr = reinterpret_cast<uint32_t*>(smem + L::taddr);
    const float* sb = reinterpret_cast<const float*>(smem + L::bias);
    const int tid = threadIdx.x, warp = tid >> 5;
    const Frame& f0 = fs.f[0];
    const uint32_t n_pix = f0.pix_all;
    const uint32_t P1 = (uint32_t)(f0.width * f0.height);
    const uint32_t n_tiles = (n_pix + kShadeThreads - 1) / kShadeThreads;

    stage_weights(smem, params);
    if (tid == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(mbar)));
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(s_taddr)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_taddr;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;   // this warp's TMEM lanes
    const uint32_t sx = smem_u32(smem + L::x), sh1 = smem_u32(smem + L::h1),
                   sh2 = smem_u32(smem + L::h2);
    const uint32_t sw1 = smem_u32(smem + L::w1), sw2 = smem_u32(smem + L::w2),
                   sw3 = smem_u32(smem + L::w3);
    uint32_t phase = 0;
    bool ok = true;

    for (uint32_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const uint32_t p = tile * kShadeThreads + tid;
        const bool valid = p < n_pix;
        // ---- layer 1 input: 16 features and the view direction, bf16
        {
            float in[kIn];
#pragma unroll
            for (int k = 0; k < kIn; ++k) in[k] = 0.0f;
            if (valid) {
                const float4* fp = reinterpret_cast<const float4*>(features + (size_t)p * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 t = fp[q];
                    in[4 * q] = t.x;
                    in[4 * q + 1] = t.y;
                    in[4 * q + 2] = t.z;
                    in[4 * q + 3] = t.w;
                }
                const uint32_t cam = p / P1;
                view_dir(fs.f[cam], p - cam * P1, in + 16);
            }
#pragma unroll
            for (int j = 0; j < kIn / 8; ++j)
                *reinterpret_cast<uint4*>(smem + L::x + kmajor_off(tid, 8 * j, kIn)) = pack8(in + 8 * j);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            for (int k0 = 0; k0 < kIn; k0 += 16)
                mma_bf16(tmem, smem_desc(sx + (k0 / 8) * 128, 128, (kIn / 8) * 128),
                         smem_desc(sw1 + (k0 / 8) * 128, 128, (kIn / 8) * 128),
                         idesc_bf16(128, kHid), k0 > 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));   // one decision for all
        ++phase;
        tc_fence_after();
        if (!ok) break;
        // ---- h1 = ReLU(D1 + b1) -> A of layer 2
#pragma unroll
        for (int c0 = 0; c0 < kHid; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j] + sb[c0 + j], 0.0f);
            *reinterpret_cast<uint4*>(smem + L::h1 + kmajor_off(tid, c0, kHid)) = pack8(v);
            *reinterpret_cast<uint4*>(smem + L::h1 + kmajor_off(tid, c0 + 8, kHid)) = pack8(v + 8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            for (int k0 = 0; k0 < kHid; k0 += 16)
                mma_bf16(tmem + kHid, smem_desc(sh1 + (k0 / 8) * 128, 128, (kHid / 8) * 128),
                         smem_desc(sw2 + (k0 / 8) * 128, 128, (kHid / 8) * 128),
                         idesc_bf16(128, kHid), k0 > 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));   // one decision for all
        ++phase;
        tc_fence_after();
        if (!ok) break;
        // ---- h2 = ReLU(D2 + b2) -> A of layer 3
#pragma unroll
        for (int c0 = 0; c0 < kHid; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(kHid + c0), v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j] + sb[kHid + c0 + j], 0.0f);
            *reinterpret_cast<uint4*>(smem + L::h2 + kmajor_off(tid, c0, kHid)) = pack8(v);
            *reinterpret_cast<uint4*>(smem + L::h2 + kmajor_off(tid, c0 + 8, kHid)) = pack8(v + 8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            for (int k0 = 0; k0 < kHid; k0 += 16)
                mma_bf16(tmem, smem_desc(sh2 + (k0 / 8) * 128, 128, (kHid / 8) * 128),
                         smem_desc(sw3 + (k0 / 8) * 128, 128, (kHid / 8) * 128),
                         idesc_bf16(128, kOutPad), k0 > 0);
            mma_commit(mbar);
        }
        ok = __syncthreads_and(mbar_wait(mbar, phase & 1));   // one decision for all
        ++phase;
        tc_fence_after();
        if (!ok) break;
        // ---- y = D3 + b3
        {
            float v[16];
            tmem_ld16(tmem + lane_base, v);
            if (valid) {
#pragma unroll
                for (int o = 0; o < 3; ++o) rgb[(size_t)p * 3 + o] = v[o] + sb[2 * kHid + o];
            }
        }
        tc_fence_before();
        __syncthreads();   // the tile's operands and accumulators are free
        tc_fence_after();
    }
    if (!ok) {
        // an MMA did not complete in time: report it, give it one more
        // bounded wait, then release the tensor memory regardless
        if (tid == 0) atomicOr(&w.state->error, kErrTimeout);
        mbar_wait(mbar, (phase - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

}  // namespace

cudaError_t prepare_shade() {
    return cudaFuncSetAttribute(k_shade_forward, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                ShadeSmem::bytes);
}

cudaError_t launch_shade_forward(const Frames& fs, const Workspace& w, const float* features,
                                 const float* params, float* rgb, int n_sms, cudaStream_t stream) {
    const uint32_t n_tiles = (fs.f[0].pix_all + kShadeThreads - 1) / kShadeThreads;
    if (n_tiles == 0) return cudaSuccess;
    const uint32_t cap = (uint32_t)(4 * n_sms);   // 4 CTAs of 128 TMEM columns fill an SM's 512
    const int grid = (int)(n_tiles < cap ? n_tiles : cap);
    k_shade_forward<<<grid, kShadeThreads, ShadeSmem::bytes, stream>>>(fs, w, features, params, rgb);
    return cudaGetLastError();
}

}  // namespace pulsar
