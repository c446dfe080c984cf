// Prompt-chunk projections on the 5th-generation tensor cores: Y = X W^T for
// up to 2,048 activation rows, with the same fused epilogues as the decode
// matvec (pull request #1415, section "How": "prompt chunks of up to 2,048
// rows on the tensor-unit GEMM").  fp32 accumulation in tensor memory, one
// rounding to bf16 per output.
//
// One CTA per SM, persistent over output tiles of 128 activation rows x 256
// weight rows (256 output features; for QKV two heads of [q | k | v], for
// SwiGLU 128 gate rows and the 128 up rows of the same features, so that every
// pair an epilogue combines lands in the same thread):
//   warp 0      TMA producer: per 64-wide k-block, the 128 x 64 activation box
//               and the N x 64 weight box(es), 128-byte swizzled, into a ring
//               of shared-memory stages;
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               (M = 128, N = 256, K = 16; four per stage) into one of two
//               accumulators and commits each stage back to the producer;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               the op after the projection, bf16 stores; the accumulator is
//               then handed back to the MMA thread, so a tile's epilogue
//               overlaps the next tile's MMAs.
// Tiles are ordered weight-tile-major so that concurrent CTAs share weight
// tiles in L2; the activation rows (<= 2,048 x K) stay L2-resident.
#include <cuda.h>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace tfl {
namespace {

constexpr int kTM = 128;           // activation rows per tile (MMA M, TMEM lanes)
constexpr int kThreads = 6 * 32;
constexpr int kABytes = kTM * 128;  // 128 rows x 64 bf16

template <int N>
struct GCfg {
    static constexpr int kBBytes = N * 128;
    static constexpr int kStage = kABytes + kBBytes;
    static constexpr int kDepth = (192 * 1024) / kStage;
    static constexpr int kTmemCols = 2 * N;  // two accumulators
    static constexpr int kSmem = 1024 + kDepth * kStage + (2 * kDepth + 4) * 8 + 64;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Global head index gh of [q heads | k heads | v heads] -> segment (0 q, 1 k, 2 v) and head.
__device__ __forceinline__ void qkv_head(const MatvecArgs& e, int gh, int& seg, int& head) {
    seg = gh < e.n_q ? 0 : (gh < e.n_q + e.n_kv ? 1 : 2);
    head = gh - (seg == 0 ? 0 : seg == 1 ? e.n_q : e.n_q + e.n_kv);
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs a) {
    using C = GCfg<N>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kDepth * C::kStage);
    uint64_t* empty = full + C::kDepth;
    uint64_t* acc_full = empty + C::kDepth;   // [2]
    uint64_t* acc_empty = acc_full + 2;       // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // MMA completion after an abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = a.m_tiles * a.n_tiles;
    const int KB = a.kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kDepth; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool mma_any = false;  // the MMA thread issued at least one MMA

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            pdl_wait();
            const uint64_t pa = policy_evict_last(), pb = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x) {
                const int n = t / a.m_tiles, m = t % a.m_tiles;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, a.status)) {
                        *s_abort = 1;
                        break;
                    }
                    unsigned char* sA = base + stage * C::kStage;
                    unsigned char* sB = sA + kABytes;
                    mbar_arrive_expect_tx(&full[stage], C::kStage);
                    tma_load_2d(sA, &a.amap, kb * 64, m * kTM, &full[stage], pa);
                    if (a.e.mode == MV_SWIGLU) {  // 128 gate rows, then the 128 up rows of the same features
                        tma_load_2d(sB, &a.bmap[0], kb * 64, n * 128, &full[stage], pb);
                        tma_load_2d(sB + 128 * 128, &a.bmap[1], kb * 64, n * 128, &full[stage], pb);
                    } else if (a.e.mode == MV_QKV_ROPE) {  // heads 2n and 2n+1 of [q heads | k heads | v heads]
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            int seg, head;
                            qkv_head(a.e, 2 * n + hh, seg, head);
                            tma_load_2d(sB + hh * 128 * 128, &a.bmap[seg], kb * 64, head * kHeadDim, &full[stage], pb);
                        }
                    } else {
                        tma_load_2d(sB, &a.bmap[0], kb * 64, n * N, &full[stage], pb);
                    }
                    ++issued;
                    if (++stage == C::kDepth) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // after an abort, the copies already issued land before the CTA exits
            if (*s_abort) drain_ring(full, C::kDepth, stage, phase, issued, a.status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTM, N);
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t acc_phase = 0;
            bool any = false;
            for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x) {
                // the epilogue must have drained this accumulator
                if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1u, a.status)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * N);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, a.status)) {
                        *s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(base + stage * C::kStage);
                    const uint32_t sB = sA + kABytes;
                    const uint64_t da = sdesc_sw128(sA), db = sdesc_sw128(sB);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 16 per MMA: +32 bytes (2 in the >>4 address field)
                        tc_mma_bf16(d, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
                    any = true;
                    tc_commit(&empty[stage]);
                    if (++stage == C::kDepth) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(&acc_full[buf]);
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            mma_any = any;
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        pdl_wait();
        const int sub = warp & 3;               // TMEM lane quarter this warp may read
        const int rowt = sub * 32 + lane;       // row within the tile
        const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
        int buf = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            // the warp leaves together (its lanes then skip whole-warp tensor-memory loads alike)
            bool stop = *s_abort != 0;
            if (!stop) stop = !mbar_wait(&acc_full[buf], acc_phase, a.status);
            if (__any_sync(0xffffffffu, stop)) {
                *s_abort = 1;
                break;
            }
            tc_fence_after();
            const int n = t / a.m_tiles, m = t % a.m_tiles;
            const int r = m * kTM + rowt;
            const bool live = r < a.e.n_rows;
            const uint32_t acc = tmem + lane_addr + (uint32_t)(buf * N);
            if (a.e.mode == MV_STORE || a.e.mode == MV_RESIDUAL) {
                for (int c = 0; c < N / 16; ++c) {
                    float v[16];
                    __syncwarp();
                    tmem_ld16(acc + c * 16, v);
                    if (!live) continue;
                    const size_t f0 = (size_t)n * N + c * 16;
                    uint4 o[2];
                    bf16* oe = reinterpret_cast<bf16*>(o);
                    if (a.e.mode == MV_RESIDUAL) {
                        uint4* hp = reinterpret_cast<uint4*>(a.e.h + (size_t)r * a.e.n_out + f0);
                        uint4 hv[2] = {hp[0], hp[1]};
                        const bf16* he = reinterpret_cast<const bf16*>(hv);
#pragma unroll
                        for (int j = 0; j < 16; ++j) oe[j] = rn(bf(he[j]) + rbf(v[j]));
                        hp[0] = o[0];
                        hp[1] = o[1];
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) oe[j] = rn(v[j]);
                        uint4* yp = reinterpret_cast<uint4*>(a.e.y + (size_t)r * a.e.ldy + f0);
                        yp[0] = o[0];
                        yp[1] = o[1];
                    }
                }
            } else if (a.e.mode == MV_SWIGLU) {
                for (int c = 0; c < 8; ++c) {
                    float gv[16], uv[16];
                    __syncwarp();
                    tmem_ld16(acc + c * 16, gv);
                    tmem_ld16(acc + 128 + c * 16, uv);
                    if (!live) continue;
                    uint4 o[2];
                    bf16* oe = reinterpret_cast<bf16*>(o);
#pragma unroll
                    for (int j = 0; j < 16; ++j) oe[j] = rn(rbf(silu_f(rbf(gv[j]))) * rbf(uv[j]));
                    uint4* yp = reinterpret_cast<uint4*>(a.e.y + (size_t)r * a.e.ldy + (size_t)n * 128 + c * 16);
                    yp[0] = o[0];
                    yp[1] = o[1];
                }
            } else {  // MV_QKV_ROPE: heads 2n, 2n+1 of [q heads | k heads | v heads]
              for (int hh = 0; hh < 2; ++hh) {
                int seg, head;
                qkv_head(a.e, 2 * n + hh, seg, head);
                const int pos = a.e.rows.pos0[0] + r;
                bf16* dst = nullptr;
                if (live) {
                    dst = seg == 0 ? a.e.y + (size_t)r * a.e.ldy + (size_t)head * kHeadDim
                                   : kv_row(a.e.rows.kv[0], a.e.layer, seg - 1, pos, a.e.n_kv) +
                                         (size_t)head * kHeadDim;
                }
                const uint32_t acc_h = acc + (uint32_t)(hh * 128);
                for (int c = 0; c < 4; ++c) {
                    float lo[16], hi[16];
                    __syncwarp();
                    tmem_ld16(acc_h + c * 16, lo);
                    tmem_ld16(acc_h + 64 + c * 16, hi);
                    if (!live) continue;
                    uint4 ol[2], oh[2];
                    bf16* ole = reinterpret_cast<bf16*>(ol);
                    bf16* ohe = reinterpret_cast<bf16*>(oh);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float xl = rbf(lo[j]), xh = rbf(hi[j]);
                        if (seg < 2) {
                            const int jl = c * 16 + j;
                            const float cs = bf(a.e.cos_t[(size_t)pos * 64 + jl]);
                            const float sn = bf(a.e.sin_t[(size_t)pos * 64 + jl]);
                            ole[j] = rn(rbf(xl * cs) + rbf(-xh * sn));
                            ohe[j] = rn(rbf(xh * cs) + rbf(xl * sn));
                        } else {
                            ole[j] = rn(xl);
                            ohe[j] = rn(xh);
                        }
                    }
                    uint4* pl = reinterpret_cast<uint4*>(dst + c * 16);
                    uint4* ph = reinterpret_cast<uint4*>(dst + 64 + c * 16);
                    pl[0] = ol[0];
                    pl[1] = ol[1];
                    ph[0] = oh[0];
                    ph[1] = oh[1];
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
        pdl_trigger();
    }

    // all MMAs were waited for by the epilogue (or, after an abort, are waited
    // for below): free TMEM
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // after an abort, every MMA already issued completes before tensor
        // memory is freed (a commit tracks all of this thread's earlier MMAs)
        if (lane == 0 && *s_abort && mma_any) {
            tc_commit(drain);
            mbar_wait(drain, 0u, a.status);
        }
        tc_fence_after();
        __syncwarp();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int N>
cudaError_t launch_n(const GemmArgs& a, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = GCfg<N>::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<N>, a);
}

}  // namespace

cudaError_t init_gemm_tc() {
    return cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, GCfg<256>::kSmem);
}

int gemm_tile_n(int) { return 256; }

int gemm_n_tiles(const MatvecArgs& e) {
    if (e.mode == MV_SWIGLU) return e.n_out % 128 == 0 ? e.n_out / 128 : -1;
    if (e.mode == MV_QKV_ROPE) return (e.n_q + 2 * e.n_kv) % 2 == 0 ? (e.n_q + 2 * e.n_kv) / 2 : -1;
    return e.n_out % 256 == 0 ? e.n_out / 256 : -1;
}

cudaError_t launch_gemm_tc(const GemmArgs& a, int grid, cudaStream_t st, bool pdl) {
    if (a.e.n_rows < 1 || a.e.n_rows > a.m_tiles * kTM || a.kblocks < 1 || a.n_tiles < 1 || a.e.K != a.kblocks * 64 ||
        a.n_tiles != gemm_n_tiles(a.e))
        return cudaErrorInvalidValue;
    const int total = a.m_tiles * a.n_tiles;
    if (grid > total) grid = total;
    return launch_n<256>(a, grid, st, pdl);
}

}  // namespace tfl
