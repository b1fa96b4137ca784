// splitk_gemm.cu -- a split-K GEMM whose epilogue applies the canonical fold
// over split ids, so that the per-split partial sums never leave the SM.
//
// The mHC backward is forced into split-K (an output 24 wide, K = 7168): each
// K-split produces its own partial and a deterministic reduce sums them in
// split-id order ("DeepSeek-V4 book, Ch 09: Batch invariance and
// determinism", section 3.3); several writers of one output element get
// private slots merged in a fixed order ("Bit-exact training interview
// notes", table "where nondeterminism comes from", the grouped-GEMM epilogue
// row).  det_splitk_reduce does that reduce over partials in memory; here the
// producer GEMM keeps each split's partial in tensor memory and folds it
// straight away:
//
//     out[r][c] = canonical sum over s = 0 .. S-1 of P_s[r][c],
//     P_s[r][c] = the tensor cores' binary32 accumulation of A[r][k] * W[c][k]
//                 over the K/S values of k in split s,
//
// with the same fold as everywhere in this library: chunks of 32 splits
// folded left to right from the first, then the level-wise pairwise tree over
// the chunk sums with the odd one carried up.
//
// One CTA owns 128 rows and all S splits.  Warp 0 streams 64-wide K blocks of
// A (128 rows) and W (32 rows, zero past C) into a ring of shared-memory
// stages with TMA (128-byte swizzle) on mbarriers, two blocks per stage fill
// where they divide a split; one thread each of warps 1 and 2 issues
// tcgen05.mma (bf16 in, fp32 accumulate, M = 128, N = 32, K = 16 each) for
// the even and the odd splits into one of four tensor-memory accumulators,
// used in turn by the splits (so the MMAs run up to four splits ahead of the
// epilogue); warps 3..6 read each finished accumulator (tcgen05.ld, one row
// per thread), release it, and fold it into the row's running chunk in split
// order.  Every wait is
// bounded; on expiry the CTA records the error, drains its own copies and
// MMAs (bounded too), frees its tensor memory and returns.
#include <cuda.h>  // CUtensorMap and the tensor-map enums (types only; entry points come from the runtime)

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace detr {

constexpr int kSgBM = 128;               // rows per CTA = tensor-memory lanes
constexpr int kSgBN = 32;                // MMA N: columns of W (C <= 32, zero past C)
constexpr int kSgBK = 64;                // K per stage: one 128-byte swizzle row of bf16
constexpr int kSgStages = 9;            // at most; fewer when the fold stack needs the room
constexpr int kSgIssuers = 2;            // MMA-issuing warps (one thread each), taking the splits in turn
constexpr int kSgThreads = 32 * (1 + kSgIssuers + 4);  // warp 0 TMA, warps 1..2 MMA (1 owns the tensor memory), 3..6 epilogue
constexpr int kSgAcc = 4;                // tensor-memory accumulators, used in turn by the splits (a power of 2)
static_assert((kSgAcc & (kSgAcc - 1)) == 0, "accumulator index by mask");
constexpr int kSgTmemCols = kSgAcc * kSgBN;  // 128 columns
constexpr int kSgMaxLevels = 4;          // fold counter levels: S <= 32 * 2^(levels - 1) = 256
constexpr uint32_t kSgABytes = kSgBM * kSgBK * 2;  // 16 KB
constexpr uint32_t kSgWBytes = kSgBN * kSgBK * 2;  // 4 KB
constexpr long long kSgPollLimit = 1ll << 24;

// Error word of the kernel (an expired wait), read by the host with
// debug_checks.  Shared by every call.
__device__ int g_sg_status;

struct SgArgs {
    int R, C, S;
    int kbs;           // K blocks of 64 per split
    int levels;        // fold counter levels
    int ns;            // shared-memory stages in use (<= kSgStages)
    void* out;
    long long ldo;
    int out_bf16;
    float* partials;   // optional: split s's partial, row-major [R][C], at partials + s * ldp
    long long ldp;
};

__device__ __forceinline__ uint32_t sg_smem(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete; false if it did not in
// time or another role gave up (*abort).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort)
{
    for (long long it = 0; it < kSgPollLimit; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 255) == 255 && *abort) return false;
    }
    return false;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile stored as TMA writes
// it with the 128-byte swizzle: rows of 128 bytes (64 values), groups of 8
// rows 1024 bytes apart.  Fields: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29; not used by swizzled K-major tiles), stride byte
// offset >> 4 (32-45: the 1024 bytes between 8-row groups), the fixed version
// 1 (46-47), base offset 0 (49-51: stages are 1024-byte aligned), swizzle
// mode 2 = 128-byte (61-63).  Successive K steps of 16 values within the 128
// bytes start 32 bytes further on.
__device__ __forceinline__ uint64_t sg_desc(uint32_t addr)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16 >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
constexpr uint32_t kSgIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kSgBN >> 3) << 17) |
                              (static_cast<uint32_t>(kSgBM >> 4) << 24);

__device__ __forceinline__ void sg_tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void sg_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kSgIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void sg_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void sg_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// KPS: K blocks per stage fill (divides kbs), a constant so that the issuing
// threads' index arithmetic stays as short as possible.
template <int KPS>
__global__ void __launch_bounds__(kSgThreads, 1)
splitk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ SgArgs a)
{
    __shared__ __align__(8) unsigned long long bar_full[kSgStages], bar_empty[kSgStages];
    __shared__ __align__(8) unsigned long long bar_tfull[kSgAcc], bar_tempty[kSgAcc], bar_drain[kSgIssuers];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    extern __shared__ __align__(1024) unsigned char sg_dyn[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t dyn = sg_smem(sg_dyn);
    const uint32_t base = (dyn + 1023u) & ~1023u;       // stages 1024-byte aligned for the swizzle
    const int NS = a.ns;
    const uint32_t sA = base;                           // NS x KPS x 16 KB
    const uint32_t sW = base + NS * KPS * kSgABytes;    // NS x KPS x 4 KB
    float* stack = reinterpret_cast<float*>(sg_dyn + (sW + NS * KPS * kSgWBytes - dyn));  // [levels][32][128]
    const int row0 = static_cast<int>(blockIdx.x) * kSgBM;
    const int nkb = a.S * a.kbs;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(sg_smem(&bar_full[i]), 1);
            mbar_init(sg_smem(&bar_empty[i]), 1);
        }
        for (int i = 0; i < kSgAcc; ++i) {
            mbar_init(sg_smem(&bar_tfull[i]), 1);
            mbar_init(sg_smem(&bar_tempty[i]), 4);  // one arrival per epilogue warp
        }
        for (int i = 0; i < kSgIssuers; ++i) mbar_init(sg_smem(&bar_drain[i]), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {  // the whole warp allocates the two accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sg_smem(&tmem_slot)),
                     "r"(kSgTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // producer: K blocks in order, split after split.  One thread issues
        // every copy, so the loop carries the stage and its phase instead of
        // dividing by the stage count.
        if (lane == 0) {
            const int nfill = nkb / KPS;
            int issued = 0;
            int st = 0, kb = 0;
            uint32_t ph = 0;  // parity of the stage's current use
            for (int f = 0; f < nfill; ++f) {
                if (f >= NS && !mbar_wait(sg_smem(&bar_empty[st]), ph ^ 1u, &abort_flag)) {
                    abort_flag = 1;
                    atomicOr(&g_sg_status, 1);
                    break;
                }
                const uint32_t bar = sg_smem(&bar_full[st]);
                mbar_expect_tx(bar, KPS * (kSgABytes + kSgWBytes));
                for (int j = 0; j < KPS; ++j, ++kb) {
                    sg_tma_2d(sA + (st * KPS + j) * kSgABytes, &tmA, kb * kSgBK, row0, bar);
                    sg_tma_2d(sW + (st * KPS + j) * kSgWBytes, &tmW, kb * kSgBK, 0, bar);
                }
                ++issued;
                if (++st == NS) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            // every copy this CTA issued has landed before it may leave
            for (int f = issued > NS ? issued - NS : 0; f < issued; ++f)
                mbar_wait(sg_smem(&bar_full[f % NS]), (f / NS) & 1, &abort_flag);
        }
    } else if (warp <= kSgIssuers) {
        // MMA issuers: split s into accumulator s % kSgAcc, issued by thread
        // 0 of warp 1 + s % kSgIssuers.  The issuing threads' loops are the
        // kernel's critical path (one thread took about 250 ns per K block
        // when it divided by the stage count and rebuilt every descriptor):
        // two of them take the splits in turn, and each carries its stage,
        // phase and descriptors (a stage's descriptors are the first stage's
        // plus its offset >> 4; each K step of 16 values adds 32 bytes, 2 in
        // the address field).  A split's fills are consecutive, and each
        // issuer skips the other's; every wait points to an earlier split, so
        // no cycle of waits can form.
        if (lane == 0) {
            const int me = warp - 1;
            bool ok = true;
            const uint64_t dA0 = sg_desc(sA), dW0 = sg_desc(sW);
            const int nfps = a.kbs / KPS;  // stage fills per split
            int st = (me * nfps) % NS, sub = 0;  // stage and K block within its fill (KPS divides kbs)
            uint32_t ph = ((me * nfps) / NS) & 1u;
            for (int s = me; s < a.S && ok; s += kSgIssuers) {
                const int buf = s & (kSgAcc - 1);
                if (s >= kSgAcc && !mbar_wait(sg_smem(&bar_tempty[buf]), ((s / kSgAcc) - 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kSgBN);
                for (int j = 0; j < a.kbs; ++j) {
                    if (sub == 0) {
                        if (!mbar_wait(sg_smem(&bar_full[st]), ph, &abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const int slot = st * KPS + sub;
                    const uint64_t dA = dA0 + static_cast<uint64_t>(slot) * (kSgABytes >> 4);
                    const uint64_t dW = dW0 + static_cast<uint64_t>(slot) * (kSgWBytes >> 4);
#pragma unroll
                    for (int k = 0; k < kSgBK / 16; ++k)
                        sg_mma(d, dA + 2 * k, dW + 2 * k, (j > 0 || k > 0) ? 1u : 0u);
                    if (++sub == KPS) {
                        sg_commit(sg_smem(&bar_empty[st]));  // the stage is free once these MMAs have read it
                        sub = 0;
                        if (++st == NS) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (ok) sg_commit(sg_smem(&bar_tfull[buf]));  // the accumulator is complete
                for (int q = 0; q < (kSgIssuers - 1) * nfps; ++q) {  // the other issuers' fills
                    if (++st == NS) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                abort_flag = 1;
                atomicOr(&g_sg_status, 1);
            }
            // every MMA this thread issued has finished before the memory is freed
            sg_commit(sg_smem(&bar_drain[me]));
            mbar_wait(sg_smem(&bar_drain[me]), 0, &abort_flag);
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const int q = warp & 3;
        const int rl = 32 * q + lane;
        const int row = row0 + rl;
        float chunk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) chunk[c] = 0.0f;
        unsigned int cnt = 0;
        bool ok = true;
        for (int s = 0; s < a.S; ++s) {
            const int buf = s % kSgAcc;
            // the warp goes on only together (tcgen05.ld is warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait(sg_smem(&bar_tfull[buf]), (s / kSgAcc) & 1, &abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[32];
            sg_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * kSgBN), v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sg_smem(&bar_tempty[buf]));
            if (a.partials && row < a.R) {
                float* p = a.partials + static_cast<long long>(s) * a.ldp + static_cast<long long>(row) * a.C;
                for (int c = 0; c < a.C; ++c) p[c] = v[c];
            }
            // fold left to right inside the chunk of 32 splits, from its first
            const bool first = (s & 31) == 0;
#pragma unroll
            for (int c = 0; c < 32; ++c) chunk[c] = first ? v[c] : __fadd_rn(chunk[c], v[c]);
            if ((s & 31) == 31 || s == a.S - 1) {
                // push the chunk sum into the binary counter (stack in shared
                // memory, one column per row): merging it with its completed
                // left neighbours is the level-wise pairwise tree
                unsigned int cc = cnt;
                int L = 0;
                while (cc & 1u) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) chunk[c] = __fadd_rn(stack[(L * 32 + c) * kSgBM + rl], chunk[c]);
                    cc >>= 1;
                    ++L;
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) stack[(L * 32 + c) * kSgBM + rl] = chunk[c];
                ++cnt;
            }
        }
        if (!ok) {
            abort_flag = 1;
            atomicOr(&g_sg_status, 1);
        } else if (row < a.R) {
            // the partial nodes at the right edge combine from the lowest level up
            float res[32];
            bool have = false;
            for (int L = 0; (cnt >> L) != 0u; ++L) {
                if ((cnt >> L) & 1u) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float x = stack[(L * 32 + c) * kSgBM + rl];
                        res[c] = have ? __fadd_rn(x, res[c]) : x;
                    }
                    have = true;
                }
            }
            if (a.out_bf16) {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + static_cast<long long>(row) * a.ldo;
                for (int c = 0; c < a.C; ++c) o[c] = __float2bfloat16_rn(res[c]);
            } else {
                float* o = static_cast<float*>(a.out) + static_cast<long long>(row) * a.ldo;
                for (int c = 0; c < a.C; ++c) o[c] = res[c];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kSgTmemCols) : "memory");
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_sg_mu;
EncodeTiled g_encode = nullptr;

det_status encode_fn(EncodeTiled* out)
{
    std::lock_guard<std::mutex> lk(g_sg_mu);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        DETR_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !f) return DET_ERR_UNSUPPORTED;
        g_encode = reinterpret_cast<EncodeTiled>(f);
    }
    *out = g_encode;
    return DET_OK;
}

// K-major bf16 matrix [rows][ld] (K = cols): boxes of 64 values x box_rows
// rows, 128-byte swizzle, zero fill past the edges.
det_status make_map(EncodeTiled enc, CUtensorMap* m, const void* p, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kSgBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DET_OK : DET_ERR_ARG;
}

int fold_levels(int S)
{
    const int nc = (S + 31) / 32;
    int L = 1;
    while ((1 << L) <= nc) ++L;  // floor(log2(nc)) + 1
    return L;
}
}  // namespace

}  // namespace detr

using namespace detr;

extern "C" det_status det_splitk_gemm_reduce(const void* A, int64_t lda, const void* W, int64_t ldw, int64_t R,
                                             int32_t C, int64_t K, int32_t S, det_dtype ab_dtype, void* out,
                                             int64_t ldo, det_dtype out_dtype, float* partials, int64_t ldp,
                                             const det_opts* opts, void* stream)
{
    if (ab_dtype != DET_BF16 || !dtype_ok(out_dtype)) return DET_ERR_DTYPE;
    if (R < 0 || K < 0 || C < 1 || S < 1 || ldo < C) return DET_ERR_ARG;
    if (C > kSgBN || S > 32 * (1 << (kSgMaxLevels - 1)) || R > kMaxRows || K > kMaxRows) return DET_ERR_UNSUPPORTED;
    if (K % S != 0 || (K / S) % kSgBK != 0 || K == 0) return DET_ERR_UNSUPPORTED;
    if (!A || !W || (R > 0 && !out)) return DET_ERR_ARG;
    if (lda < K || ldw < K || !aligned(A, 16) || !aligned(W, 16) || (lda * 2) % 16 != 0 || (ldw * 2) % 16 != 0)
        return DET_ERR_ARG;
    const int osz = dtype_size(out_dtype);
    if (!aligned(out, static_cast<size_t>(osz)) || (partials && (!aligned(partials, 4) || ldp < R * C)))
        return DET_ERR_ARG;
    const size_t out_bytes = R > 0 ? static_cast<size_t>((R - 1) * ldo + C) * osz : 0;
    if (overlaps(out, out_bytes, A, static_cast<size_t>(R > 0 ? (R - 1) * lda + K : 0) * 2) ||
        overlaps(out, out_bytes, W, static_cast<size_t>((C - 1) * ldw + K) * 2) ||
        (partials && overlaps(out, out_bytes, partials, static_cast<size_t>((S - 1) * ldp + R * C) * 4)))
        return DET_ERR_ARG;
    if (opts && opts->reserved[0]) return DET_ERR_ARG;
    if (R == 0) return DET_OK;
    EncodeTiled enc = nullptr;
    det_status s = encode_fn(&enc);
    if (s) return s;
    CUtensorMap mA, mW;
    s = make_map(enc, &mA, A, R, K, lda, kSgBM);
    if (s) return s;
    s = make_map(enc, &mW, W, C, K, ldw, kSgBN);
    if (s) return s;
    SgArgs a{};
    a.R = static_cast<int>(R);
    a.C = C;
    a.S = S;
    a.kbs = static_cast<int>((K / S) / kSgBK);
    a.levels = fold_levels(S);
    a.out = out;
    a.ldo = ldo;
    a.out_bf16 = out_dtype == DET_BF16 ? 1 : 0;
    a.partials = partials;
    a.ldp = ldp;
    // two K blocks per stage fill where a split has an even number of them
    // (half the barrier round trips of the issuing threads), and as many
    // stages as fit beside the fold stack (227 KB per CTA at most)
    const int kps = a.kbs % 2 == 0 ? 2 : 1;
    const size_t stack = static_cast<size_t>(a.levels) * 32 * kSgBM * sizeof(float);
    const size_t room = size_t(227) * 1024 - 2048 - 1024 - stack;
    const size_t fill = static_cast<size_t>(kps) * (kSgABytes + kSgWBytes);
    a.ns = static_cast<int>(std::min<size_t>(kSgStages, room / fill));
    if (a.ns < 2) return DET_ERR_UNSUPPORTED;
    const size_t smem = 1024 + static_cast<size_t>(a.ns) * fill + stack;
    const void* kern = kps == 2 ? reinterpret_cast<const void*>(splitk_gemm_kernel<2>)
                                : reinterpret_cast<const void*>(splitk_gemm_kernel<1>);
    s = allow_dynamic_smem(kern, smem);
    if (s) return s;
    cudaStream_t st = as_stream(stream);
    const unsigned int grid = static_cast<unsigned int>(cdiv(R, kSgBM));
    if (kps == 2) splitk_gemm_kernel<2><<<grid, kSgThreads, smem, st>>>(mA, mW, a);
    else splitk_gemm_kernel<1><<<grid, kSgThreads, smem, st>>>(mA, mW, a);
    DETR_LAUNCHED();
    if (opts && opts->debug_checks) {
        DETR_CUDA(cudaStreamSynchronize(st));
        int h = 0;
        DETR_CUDA(cudaMemcpyFromSymbol(&h, g_sg_status, sizeof(int)));
        if (h) {
            const int zero = 0;
            DETR_CUDA(cudaMemcpyToSymbol(g_sg_status, &zero, sizeof(int)));
            return DET_ERR_TIMEOUT;
        }
    }
    return DET_OK;
}
