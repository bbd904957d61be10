// Small pieces of the chunk form of the gated delta rule shared by the two
// chunked-prefill kernels (tensor-core and plain fp32): the in-chunk cumulative
// log-decay, the gate exponential and the unit lower-triangular inverse
// T = (I + A)^{-1} of the WY/UT representation.
#pragma once

#include "common.cuh"

namespace chunkmath {

// G[t] = g[0] + ... + g[t] over the chunk (g = 0 past its n tokens), by one
// warp with a shuffle scan; in place allowed.
__device__ __forceinline__ void chunk_cumsum(const float *g, int n, float *G) {
    const int lane = threadIdx.x & 31;
    const float g0 = 2 * lane < n ? g[2 * lane] : 0.f;
    const float g1 = 2 * lane + 1 < n ? g[2 * lane + 1] : 0.f;
    const float pair = g0 + g1;
    float incl = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - pair;
    __syncwarp();
    G[2 * lane] = excl + g0;
    G[2 * lane + 1] = excl + pair;
}

// e^x for the gates inside a chunk (x <= 0): 2^(x log2 e) by the hardware's
// base-2 exponential (relative error about 2^-22).
__device__ __forceinline__ float gate_exp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// T = (I + A)^{-1} in place (64 x 64 fp32, row stride kAs; A strictly lower
// triangular with zeros on and above the diagonal).
// The four 16 x 16 diagonal blocks by forward substitution (one thread per
// column, rows read as float4), then the blocks below them from the block
// identities of a unit lower-triangular inverse, T_ba = -T_bb A_ba T_aa: for
// the 16-row pairs (1,0) and (3,2), then for the 32-row halves.  X: 4.5 KB.
// NT threads (256 or 512) call it; sync() is their barrier.
template <int NT, int kAs, typename Sync>
__device__ void solve_unit_lower(float *Af, float *X, int tid, Sync sync) {
    if (tid < 64) {
        const int I = tid >> 4, j = tid & 15;
        const float *Ab = Af + (16 * I) * kAs + 16 * I;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == j ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; q < (r + 3) / 4; ++q) {
                const float4 a4 = *reinterpret_cast<const float4 *>(Ab + r * kAs + 4 * q);
                if (4 * q + 0 < r) acc = fmaf(-a4.x, x[4 * q + 0], acc);
                if (4 * q + 1 < r) acc = fmaf(-a4.y, x[4 * q + 1], acc);
                if (4 * q + 2 < r) acc = fmaf(-a4.z, x[4 * q + 2], acc);
                if (4 * q + 3 < r) acc = fmaf(-a4.w, x[4 * q + 3], acc);
            }
            x[r] = acc;
        }
        __syncwarp();  // the block's A entries are read before its T column is written
#pragma unroll
        for (int r = 0; r < 16; ++r) Af[(16 * I + r) * kAs + 16 * I + j] = x[r];
    }
    sync();
    float accs[512 / NT];
#pragma unroll
    for (int u = 0; u < 512 / NT; ++u) {
        const int e = tid + u * NT;
        const int p = e >> 8, r = (e >> 4) & 15, j = e & 15;
        const int R0 = 32 * p + 16, C0 = 32 * p;
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a4 = *reinterpret_cast<const float4 *>(Af + (R0 + r) * kAs + C0 + 4 * q);
            acc = fmaf(a4.x, Af[(C0 + 4 * q + 0) * kAs + C0 + j], acc);
            acc = fmaf(a4.y, Af[(C0 + 4 * q + 1) * kAs + C0 + j], acc);
            acc = fmaf(a4.z, Af[(C0 + 4 * q + 2) * kAs + C0 + j], acc);
            acc = fmaf(a4.w, Af[(C0 + 4 * q + 3) * kAs + C0 + j], acc);
        }
        X[p * 256 + r * 16 + j] = acc;
    }
    sync();
#pragma unroll
    for (int u = 0; u < 512 / NT; ++u) {
        const int e = tid + u * NT;
        const int p = e >> 8, r = (e >> 4) & 15, j = e & 15;
        const int R0 = 32 * p + 16;
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 b4 = *reinterpret_cast<const float4 *>(Af + (R0 + r) * kAs + R0 + 4 * q);
            t = fmaf(b4.x, X[p * 256 + (4 * q + 0) * 16 + j], t);
            t = fmaf(b4.y, X[p * 256 + (4 * q + 1) * 16 + j], t);
            t = fmaf(b4.z, X[p * 256 + (4 * q + 2) * 16 + j], t);
            t = fmaf(b4.w, X[p * 256 + (4 * q + 3) * 16 + j], t);
        }
        accs[u] = -t;
    }
#pragma unroll
    for (int u = 0; u < 512 / NT; ++u) {
        const int e = tid + u * NT;
        const int p = e >> 8, r = (e >> 4) & 15, j = e & 15;
        Af[(32 * p + 16 + r) * kAs + 32 * p + j] = accs[u];
    }
    sync();
    if (tid < 256) {
        // the lower half: row 32 + r (r = lane) by warp cg for columns 4 cg ..
        // 4 cg + 3, with T's upper zeros skipped in the first product; X rows
        // padded to 36 floats so that the lanes' float4 rows use all banks
        const int r = tid & 31, cg = tid >> 5;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = cg; q < 8; ++q) {
            const float4 a4 = *reinterpret_cast<const float4 *>(Af + (32 + r) * kAs + 4 * q);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const float4 tv = *reinterpret_cast<const float4 *>(Af + (4 * q + z) * kAs + 4 * cg);
                acc.x = fmaf(av[z], tv.x, acc.x);
                acc.y = fmaf(av[z], tv.y, acc.y);
                acc.z = fmaf(av[z], tv.z, acc.z);
                acc.w = fmaf(av[z], tv.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(X + r * 36 + 4 * cg) = acc;
    }
    sync();
    if (tid < 256) {
        const int r = tid & 31, cg = tid >> 5;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 b4 = *reinterpret_cast<const float4 *>(Af + (32 + r) * kAs + 32 + 4 * q);
            const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const float4 xv = *reinterpret_cast<const float4 *>(X + (4 * q + z) * 36 + 4 * cg);
                t.x = fmaf(bv[z], xv.x, t.x);
                t.y = fmaf(bv[z], xv.y, t.y);
                t.z = fmaf(bv[z], xv.z, t.z);
                t.w = fmaf(bv[z], xv.w, t.w);
            }
        }
        *reinterpret_cast<float4 *>(Af + (32 + r) * kAs + 4 * cg) = make_float4(-t.x, -t.y, -t.z, -t.w);
    }
    sync();
}

}  // namespace chunkmath
