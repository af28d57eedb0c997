// mma_peak.cu -- FP8 tensor-core throughput probe for the roofline of the
// prefill kernels (built as libfp8kv_probe.so, loaded by the benchmark only).
//
// One CTA per SM; `issuers` threads (in different warps) each issue
// tcgen05 kind::f8f6f4 MMAs of M = 128, N = n, K = 32 (e4m3 x e4m3 -> fp32)
// back to back from shared-memory operands, cycling over `accs` TMEM
// accumulators of their own (consecutive MMAs of a thread go to different
// accumulators when accs > 1).  The operands' values do not matter for the
// rate.  FLOP = 2 * 128 * n * 32 per MMA.  `mode` picks the operands:
//   0  A and B from the same shared-memory slice every time;
//   1  A and B walk the four 32-byte K slices of their 128-byte rows;
//   2  A from tensor memory (columns 480..511, the four K slices), B as in 1;
//   3, 4, 5  as 0, 1, 2, but the issuer's whole warp runs the loop and one
//            lane, chosen by elect.sync, issues each MMA and commit;
//   6  kind::f16 (bf16 x bf16 -> fp32, K = 16) MMAs, operands as in 0, for
//      comparison (the FLOP count printed by the caller assumes K = 32);
//   7  as 1, with the loop unrolled by four over operands held in registers
//      that the loop never writes (accumulate always on).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../csrc/common.cuh"

namespace {
using namespace fp8kv;

constexpr int kCommitEvery = 64;

// clock64 stamps of CTA 0's first issuer: cycles to issue its first
// kCommitEvery MMAs, cycles from its first issue to its last completion
__device__ long long g_probe_stamps[3];

__device__ __forceinline__ void mma_bf16_probe(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__global__ void __launch_bounds__(256, 1) mma_peak_kernel(int32_t iters, int32_t n, int32_t accs,
                                                          int32_t issuers, int32_t mode,
                                                          uint32_t *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *a_tile = smem;                  // 128 rows x 128 bytes
    uint8_t *b_tile = smem + 128 * 128;      // up to 256 rows x 128 bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 128 * 128 + 256 * 128);   // [issuer][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    CtaFail *fail = reinterpret_cast<CtaFail *>(bars + 17);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (128 + 256) * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 16; ++i) mbar_init(&bars[i], 1);
        fail->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int issuer = warp;   // lane 0 (or the elected lane) of warps 0 .. issuers - 1
    const bool whole_warp = mode >= 3 && mode <= 5;
    const bool bf16 = mode == 6;
    const int opnd = bf16 ? 0 : mode % 3;
    if (((threadIdx.x & 31) == 0 || whole_warp) && issuer < issuers) {
        uint64_t *bar = bars + 2 * issuer;
        // this issuer's accumulators: n columns each, after the other issuers'
        const uint32_t acc0 = tmem + static_cast<uint32_t>(issuer * accs * n);
        const uint32_t idesc = bf16 ? (idesc_e4m3_f32(128, n, false, false) | (1u << 7) | (1u << 10))
                                    : idesc_e4m3_f32(128, n, false, false);
        const uint64_t a = sdesc_sw128(smem_u32(a_tile), 16, 1024);
        const uint64_t b = sdesc_sw128(smem_u32(b_tile), 16, 1024);
        // MMAs in batches of kCommitEvery, batch j committed to barrier j % 2
        // (phase j / 2 of it); before batch j + 2 reuses the barrier, batch j
        // is waited for, so each wait is for the newest phase of its barrier
        int32_t batches = 0;
        bool ok = true;
        auto commit_batch = [&]() {
            if (batches >= 2 && ok)
                ok = mbar_wait(&bar[batches & 1], ((batches - 2) >> 1) & 1, fail, err);
            if (whole_warp) ok = __all_sync(0xffffffffu, ok);   // keep the warp converged
            if (!whole_warp || elect_one()) tc_commit(&bar[batches & 1]);
            if (whole_warp) __syncwarp();
            ++batches;
        };
        const long long t0 = clock64();
        if (mode == 7) {
            const uint32_t d = acc0;
            const uint64_t a0 = a, a1 = a + 2u, a2 = a + 4u, a3 = a + 6u;
            const uint64_t b0 = b, b1 = b + 2u, b2 = b + 4u, b3 = b + 6u;
            for (int32_t i = 0; i < iters && ok; i += 4) {
                {
                    mma_e4m3(d, a0, b0, idesc, 1u);
                    mma_e4m3(d, a1, b1, idesc, 1u);
                    mma_e4m3(d, a2, b2, idesc, 1u);
                    mma_e4m3(d, a3, b3, idesc, 1u);
                }
                if (i == 0 && blockIdx.x == 0 && issuer == 0) g_probe_stamps[2] = clock64() - t0;
                if (i + 4 == kCommitEvery && blockIdx.x == 0 && issuer == 0)
                    g_probe_stamps[0] = clock64() - t0;
                if ((i + 4) % kCommitEvery == 0) commit_batch();
            }
        }
        for (int32_t i = 0; i < iters && ok && mode != 7; ++i) {
            const int32_t slot = i % accs;
            const uint32_t ks = opnd == 0 ? 0u : static_cast<uint32_t>(i & 3);
            if (!whole_warp || elect_one()) {
                if (bf16)
                    mma_bf16_probe(acc0 + slot * n, a, b, idesc, i >= accs ? 1u : 0u);
                else if (opnd == 2)
                    mma_e4m3_tmem_a(acc0 + slot * n, tmem + 480u + 8u * ks, b + 2u * ks, idesc,
                                    i >= accs ? 1u : 0u);
                else
                    mma_e4m3(acc0 + slot * n, a + 2u * ks, b + 2u * ks, idesc,
                             i >= accs ? 1u : 0u);
            }
            if (whole_warp) __syncwarp();
            if (i + 1 == kCommitEvery && blockIdx.x == 0 && issuer == 0 && (threadIdx.x & 31) == 0)
                g_probe_stamps[0] = clock64() - t0;
            if ((i + 1) % kCommitEvery == 0) commit_batch();
        }
        commit_batch();
        // drain the (at most two) batches not waited for (bounded)
        for (int32_t j = batches >= 2 ? batches - 2 : 0; j < batches; ++j) {
            CtaFail never{0};
            mbar_wait(&bar[j & 1], (j >> 1) & 1, &never, err);
        }
        if (blockIdx.x == 0 && issuer == 0 && (threadIdx.x & 31) == 0)
            g_probe_stamps[1] = clock64() - t0;
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}
}  // namespace

__device__ uint32_t g_probe_err;

// Times one launch of `ctas` CTAs whose `issuers` threads each issue `iters`
// MMAs of N = n over `accs` accumulators (after a shorter warm-up launch);
// *ms_out is its duration on `stream` (CUDA events).  issuers * accs * n
// columns must fit the 512 of tensor memory.  The dynamic shared memory is
// sized so that one CTA fits per SM.  Returns 0, 1 for bad arguments, 5 for
// a CUDA error, 6 if a wait ran out.
extern "C" int fp8kv_probe_mma_e4m3_mode(int32_t ctas, int32_t iters, int32_t n, int32_t accs,
                                         int32_t issuers, int32_t mode, float *ms_out,
                                         void *stream) {
    if (ctas <= 0 || iters <= 0 || (n != 64 && n != 128 && n != 256) || !ms_out || accs < 1 ||
        issuers < 1 || issuers > 8 || mode < 0 || mode > 7 || (mode == 7 && (accs != 1 || iters % 4)) ||
        issuers * accs * n > ((mode == 2 || mode == 5) ? 480 : 512))
        return 1;
    uint32_t *err = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_probe_err) != cudaSuccess) return 5;
    cudaMemset(err, 0, sizeof(uint32_t));
    const int smem = 120 * 1024;   // > half the SM's shared memory: one CTA per SM
    if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 5;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    mma_peak_kernel<<<ctas, 256, smem, s>>>(iters / 4 > 0 ? iters / 4 : 1, n, accs, issuers, mode,
                                            err);
    cudaEventRecord(e0, s);
    mma_peak_kernel<<<ctas, 256, smem, s>>>(iters, n, accs, issuers, mode, err);
    cudaEventRecord(e1, s);
    const cudaError_t st = cudaEventSynchronize(e1);
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != cudaSuccess || cudaGetLastError() != cudaSuccess) return 5;
    uint32_t e = 0;
    cudaMemcpy(&e, err, sizeof e, cudaMemcpyDeviceToHost);
    *ms_out = ms;
    return e ? 6 : 0;
}

extern "C" int fp8kv_probe_mma_e4m3(int32_t ctas, int32_t iters, int32_t n, int32_t accs,
                                    int32_t issuers, float *ms_out, void *stream) {
    return fp8kv_probe_mma_e4m3_mode(ctas, iters, n, accs, issuers, 0, ms_out, stream);
}

// The stamps of the last probe launch (see g_probe_stamps; the third is
// the cycles to issue the first four MMAs of mode 7); 0 or 5.
extern "C" int fp8kv_probe_stamps(long long *out2) {
    return cudaMemcpyFromSymbol(out2, g_probe_stamps, 3 * sizeof(long long)) == cudaSuccess ? 0 : 5;
}
