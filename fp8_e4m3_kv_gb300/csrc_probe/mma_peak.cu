// mma_peak.cu -- FP8 tensor-core throughput probe for the roofline of the
// prefill kernels (built as libfp8kv_probe.so, loaded by the benchmark only).
//
// One CTA per SM; `issuers` threads (in different warps) each issue
// tcgen05 kind::f8f6f4 MMAs of M = 128, N = n, K = 32 (e4m3 x e4m3 -> fp32)
// back to back from shared-memory operands, cycling over `accs` TMEM
// accumulators of their own (consecutive MMAs of a thread go to different
// accumulators when accs > 1).  The operands' values do not matter for the
// rate.  FLOP = 2 * 128 * n * 32 per MMA.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../csrc/common.cuh"

namespace {
using namespace fp8kv;

constexpr int kCommitEvery = 64;

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int32_t iters, int32_t n, int32_t accs,
                                                          int32_t issuers, uint32_t *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *a_tile = smem;                  // 128 rows x 128 bytes
    uint8_t *b_tile = smem + 128 * 128;      // up to 256 rows x 128 bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 128 * 128 + 256 * 128);   // [issuer][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 8);
    CtaFail *fail = reinterpret_cast<CtaFail *>(bars + 9);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (128 + 256) * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bars[i], 1);
        fail->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int issuer = warp;   // lane 0 of warps 0 .. issuers - 1
    if ((threadIdx.x & 31) == 0 && issuer < issuers) {
        uint64_t *bar = bars + 2 * issuer;
        // this issuer's accumulators: n columns each, after the other issuers'
        const uint32_t acc0 = tmem + static_cast<uint32_t>(issuer * accs * n);
        const uint32_t idesc = idesc_e4m3_f32(128, n, false, false);
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
            tc_commit(&bar[batches & 1]);
            ++batches;
        };
        for (int32_t i = 0; i < iters && ok; ++i) {
            const int32_t slot = i % accs;
            mma_e4m3(acc0 + slot * n, a, b, idesc, i >= accs ? 1u : 0u);
            if ((i + 1) % kCommitEvery == 0) commit_batch();
        }
        commit_batch();
        // drain the (at most two) batches not waited for (bounded)
        for (int32_t j = batches >= 2 ? batches - 2 : 0; j < batches; ++j) {
            CtaFail never{0};
            mbar_wait(&bar[j & 1], (j >> 1) & 1, &never, err);
        }
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
extern "C" int fp8kv_probe_mma_e4m3(int32_t ctas, int32_t iters, int32_t n, int32_t accs,
                                    int32_t issuers, float *ms_out, void *stream) {
    if (ctas <= 0 || iters <= 0 || (n != 64 && n != 128 && n != 256) || !ms_out || accs < 1 ||
        issuers < 1 || issuers > 4 || issuers * accs * n > 512)
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
    mma_peak_kernel<<<ctas, 128, smem, s>>>(iters / 4 > 0 ? iters / 4 : 1, n, accs, issuers, err);
    cudaEventRecord(e0, s);
    mma_peak_kernel<<<ctas, 128, smem, s>>>(iters, n, accs, issuers, err);
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
