// reduce_common.cuh -- device helpers shared by the gather-reduce kernels:
// row loaders, output stores and the binary counter that applies the
// level-wise pairwise tree over aligned tree nodes.
#pragma once

#include "common.cuh"

namespace detr {

template <typename XT, bool VECTOR>
struct Loader;

template <>
struct Loader<float, true> {
    static constexpr int VEC = 4;
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const unsigned char* p) { return ld_stream_v4(p); }
    static __device__ __forceinline__ void expand(const Raw& r, float* f)
    {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
};

template <>
struct Loader<uint16_t, true> {
    static constexpr int VEC = 8;
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const unsigned char* p) { return ld_stream_v4(p); }
    static __device__ __forceinline__ void expand(const Raw& r, float* f)
    {
        f[0] = bf16lo(r.x); f[1] = bf16hi(r.x); f[2] = bf16lo(r.y); f[3] = bf16hi(r.y);
        f[4] = bf16lo(r.z); f[5] = bf16hi(r.z); f[6] = bf16lo(r.w); f[7] = bf16hi(r.w);
    }
};

template <>
struct Loader<float, false> {
    static constexpr int VEC = 1;
    using Raw = float;
    static __device__ __forceinline__ Raw load(const unsigned char* p) { return __ldg(reinterpret_cast<const float*>(p)); }
    static __device__ __forceinline__ void expand(const Raw& r, float* f) { f[0] = r; }
};

template <>
struct Loader<uint16_t, false> {
    static constexpr int VEC = 1;
    using Raw = unsigned short;
    static __device__ __forceinline__ Raw load(const unsigned char* p)
    {
        return __ldg(reinterpret_cast<const unsigned short*>(p));
    }
    static __device__ __forceinline__ void expand(const Raw& r, float* f)
    {
        f[0] = __uint_as_float(static_cast<uint32_t>(r) << 16);
    }
};

// Store VEC fp32 values as OT (binary32, or bf16 rounded to nearest even).
template <typename OT, int VEC>
__device__ __forceinline__ void store_out(void* base, long long off, const float* v, bool vec)
{
    if (sizeof(OT) == 4) {
        float* o = static_cast<float*>(base) + off;
        if (vec && VEC % 4 == 0) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4)
                *reinterpret_cast<float4*>(o + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = v[e];
        }
    } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(base) + off;
        if (vec && VEC == 8) {
            uint4 pk;
            __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]);
            __nv_bfloat162 t1 = __floats2bfloat162_rn(v[2], v[3]);
            __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]);
            __nv_bfloat162 t3 = __floats2bfloat162_rn(v[6], v[7]);
            pk.x = *reinterpret_cast<uint32_t*>(&t0);
            pk.y = *reinterpret_cast<uint32_t*>(&t1);
            pk.z = *reinterpret_cast<uint32_t*>(&t2);
            pk.w = *reinterpret_cast<uint32_t*>(&t3);
            *reinterpret_cast<uint4*>(o) = pk;
        } else if (vec && VEC == 4) {
            uint2 pk;
            __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]);
            __nv_bfloat162 t1 = __floats2bfloat162_rn(v[2], v[3]);
            pk.x = *reinterpret_cast<uint32_t*>(&t0);
            pk.y = *reinterpret_cast<uint32_t*>(&t1);
            *reinterpret_cast<uint2*>(o) = pk;
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = __float2bfloat16_rn(v[e]);
        }
    }
}

// Add VEC fp32 values to the OT values already in out and store the sums
// (index_add_ semantics): out = OT(fl32(out + v)); bf16 reads back exactly.
template <typename OT, int VEC>
__device__ __forceinline__ void add_store_out(void* base, long long off, const float* v, bool vec)
{
    float old[VEC];
    if (sizeof(OT) == 4) {
        const float* o = static_cast<const float*>(base) + off;
        if (vec && VEC % 4 == 0) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
                const float4 t = *reinterpret_cast<const float4*>(o + e);
                old[e] = t.x; old[e + 1] = t.y; old[e + 2] = t.z; old[e + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) old[e] = o[e];
        }
    } else {
        const unsigned short* o = static_cast<const unsigned short*>(base) + off;
#pragma unroll
        for (int e = 0; e < VEC; ++e) old[e] = __uint_as_float(static_cast<uint32_t>(o[e]) << 16);
    }
    float sum[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) sum[e] = __fadd_rn(old[e], v[e]);
    store_out<OT, VEC>(base, off, sum, vec);
}

// Packed FP32 add (sm_100 and later): one instruction performs two IEEE
// binary32 adds, each rounded to nearest even on its own, so the bits equal
// those of two __fadd_rn.  Measured on this GPU over 2^21 random pairs: equal
// bits.  The weight multiply stays scalar (__fmul_rn): a packed multiply
// feeding a packed add was measured to be contracted into a fused
// multiply-add by the assembler, which would change the bits.
__device__ __forceinline__ unsigned long long pack2(float a, float b)
{
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float& a, float& b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ unsigned long long add2_rn(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// One term of the left-to-right fold on VEC elements: p = fl32(w * x) (no
// multiply without weights), then acc = p for the chunk's first term, else
// acc = fl32(acc + p).
template <int VEC>
__device__ __forceinline__ void fold_term(float* acc, const float* xf, bool has_w, float wv, bool first)
{
    float p[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) p[e] = has_w ? __fmul_rn(wv, xf[e]) : xf[e];
    if (first) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = p[e];
    } else if (VEC % 2 == 0) {
#pragma unroll
        for (int e = 0; e < VEC; e += 2)
            unpack2(add2_rn(pack2(acc[e], acc[(e + 1) % VEC]), pack2(p[e], p[(e + 1) % VEC])), acc[e],
                    acc[(e + 1) % VEC]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], p[e]);
    }
}

// Binary counter over aligned tree nodes: pushing node number `cnt` merges it
// with its completed left neighbours, exactly as the level-wise tree pairs them.
template <int DR, int VEC>
__device__ __forceinline__ void counter_push(float (&stk)[DR][VEC], unsigned int cnt, float* node)
{
    unsigned int c = cnt;
    bool placed = false;
#pragma unroll
    for (int L = 0; L < DR; ++L) {
        if (!placed) {
            if (c & 1u) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) node[e] = __fadd_rn(stk[L][e], node[e]);
                c >>= 1;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) stk[L][e] = node[e];
                placed = true;
            }
        }
    }
}

// After the last push: the partial nodes at the right edge are carried up,
// so the remaining levels combine from the lowest (rightmost) upward.
template <int DR, int VEC>
__device__ __forceinline__ void counter_collapse(const float (&stk)[DR][VEC], unsigned int cnt, float* res)
{
    bool have = false;
#pragma unroll
    for (int L = 0; L < DR; ++L) {
        if ((cnt >> L) & 1u) {
            if (!have) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) res[e] = stk[L][e];
                have = true;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) res[e] = __fadd_rn(stk[L][e], res[e]);
            }
        }
    }
}

// The same binary counter with its stack in shared memory: each thread owns
// a column (`col` of `ncol`), laid out [level][element][column] so that the
// accesses of a warp are conflict-free.  Pushes happen once per round, so a
// short dynamic loop costs little.
__device__ __forceinline__ float* scounter_slot(float* st, int L, int e, int VEC, int ncol, int col)
{
    return st + (static_cast<size_t>(L) * VEC + e) * ncol + col;
}

template <int VEC>
__device__ __forceinline__ void scounter_push(float* st, int ncol, int col, unsigned int cnt, float* node)
{
    unsigned int c = cnt;
    int L = 0;
    while (c & 1u) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) node[e] = __fadd_rn(*scounter_slot(st, L, e, VEC, ncol, col), node[e]);
        c >>= 1;
        ++L;
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) *scounter_slot(st, L, e, VEC, ncol, col) = node[e];
}

template <int VEC>
__device__ __forceinline__ void scounter_collapse(float* st, int ncol, int col, unsigned int cnt, float* res)
{
    bool have = false;
    for (int L = 0; (cnt >> L) != 0u; ++L) {
        if ((cnt >> L) & 1u) {
            if (!have) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) res[e] = *scounter_slot(st, L, e, VEC, ncol, col);
                have = true;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) res[e] = __fadd_rn(*scounter_slot(st, L, e, VEC, ncol, col), res[e]);
            }
        }
    }
}

}  // namespace detr
