// route_impl.cuh -- the router's block computation, shared by the standalone
// router kernel and the fused persistent layer kernel.
//
// Gate logits are fp32 in one fixed order, reproduced bit for bit by the CPU
// oracle: 32 interleaved partial sums s_j over i = j, j+32, ... (fused
// multiply-add, round to nearest), then s_j += s_{j+off} for
// off = 16, 8, 4, 2, 1, then + bias[e].  The pages name routing as the first
// step of the layer (mKernel README, kernel table, row "MoE Dispatch + FFN +
// Combine": "routes tokens to their expert ranks") but leave its arithmetic
// open; the order is fixed because the logits decide integers.
#pragma once

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace route_detail {

constexpr int kTE = 8;       // experts per warp tile
constexpr int kKC = 256;     // K elements per pipeline stage (8 chain steps)
constexpr int kStages = 3;   // cp.async pipeline depth
constexpr int kXPad = 64;    // bytes of padding per staged x row (bank spread)

// One level of the transpose-reduction on float2 accumulators: lanes L and
// L^off (same half-warp) exchange halves of their pair lists; each adds the
// partner's copy of the half it keeps (fp32 adds, element by element).
template <int HALF, int NP>
__device__ __forceinline__ void reduce_level2(float2 (&acc)[NP], int lane, int off) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int q = 0; q < HALF; ++q) {
        const float2 send = upper ? acc[q] : acc[q + HALF];
        const float2 keep = upper ? acc[q + HALF] : acc[q];
        float2 recv;
        recv.x = __shfl_xor_sync(0xffffffffu, send.x, off);
        recv.y = __shfl_xor_sync(0xffffffffu, send.y, off);
        acc[q] = make_float2(__fadd_rn(keep.x, recv.x), __fadd_rn(keep.y, recv.y));
    }
}

// Block shape: WT x WE warps; each warp owns 2*HT tokens x 8 experts (HT
// tokens per half-warp).  MINB blocks are meant to share an SM.
template <int WT, int WE, int HT, int MINB>
struct RouteTile {
    static constexpr int kTT = 2 * HT;                // tokens per warp tile
    static constexpr int kHP = HT * kTE;              // pairs per half-warp
    static constexpr int CT = kTT * WT;               // tokens per block
    static constexpr int CE = kTE * WE;               // experts per block
    static constexpr int XROW = kKC * 2 + kXPad;      // bytes per staged x row
    static constexpr int XB = CT * XROW;              // bytes of x per stage
    static constexpr int WB = CE * kKC * 4;           // bytes of Wg per stage
    static constexpr int SB = XB + WB;
    static constexpr int SMEM = kStages * SB;
};

// Gate logits of a (CT tokens) x (CE experts) block.
//
// Chain layout: lane L of a warp works in half h = L / 16 with index
// c = L % 16 and carries the chains of classes 2c and 2c+1 (columns
// i = 2c + 32m and 2c + 1 + 32m, m = 0, 1, ...) for the half's 64 pairs:
// tokens 2a + h (a = 0..7) of the warp's 16, times the warp's 8 experts.
// One 32-bit shared load gives a token's two bf16 columns, one 64-bit load
// the matching two Wg columns, and one packed fp32x2 FMA advances both chains
// (each element a correctly rounded fma, the same bits as a scalar fmaf).
// x and Wg chunks of 256 columns stream through a 3-stage cp.async ring.
// Logits of one (CT tokens) x (CE experts) block: token group tg, expert
// group eg; uses RT::SMEM bytes of shared memory at `smem` and threads
// 0..255 of the calling block (all of them must call).
template <int WT, int WE, int HT, int MINB>
__device__ __forceinline__ void route_block(uint8_t* smem, const uint16_t* __restrict__ x,
                                            const float* __restrict__ wg, const float* __restrict__ bias, int T,
                                            int d, int E, float* __restrict__ logits, int tg, int eg) {
    static_assert(WT * WE == 8, "8 warps per block");
    using RT = RouteTile<WT, WE, HT, MINB>;
    constexpr int kTT = RT::kTT;
    constexpr int kHP = RT::kHP;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int half = lane >> 4;
    const int c = lane & 15;
    const int wt = warp / WE;
    const int we = warp % WE;
    const int ct0 = tg * RT::CT;
    const int ce0 = eg * RT::CE;
    const int nk = (d + kKC - 1) / kKC;

    // Full blocks (every row in range) stream full chunks with a fixed
    // per-thread progression: x piece (row warp + 8i, 16-byte column lane),
    // Wg piece (row tid/64 + 4i, column tid%64).  Blocks at the token or expert
    // edge, and the last partial chunk, use the general loader, which clamps
    // rows past the end to the last row (loaded, never stored).
    static_assert(RT::CT % 8 == 0 && (RT::CE * (kKC / 4)) % 256 == 0, "loader shape");
    const bool full_block = (ct0 + RT::CT <= T) && (ce0 + RT::CE <= E);
    const uint16_t* xsrc = x + static_cast<int64_t>(ct0 + warp) * d + lane * 8;
    const int wr = tid / (kKC / 4), wq = tid % (kKC / 4);
    const float* wsrc = wg + static_cast<int64_t>(ce0 + wr) * d + wq * 4;
    auto load_stage = [&](int stage, int k0) {
        uint8_t* sx = smem + stage * RT::SB;
        uint8_t* sw = sx + RT::XB;
        const int kc = min(kKC, d - k0);
        if (full_block && kc == kKC) {
#pragma unroll
            for (int i = 0; i < RT::CT / 8; ++i)
                cp_async16(sx + (warp + 8 * i) * RT::XROW + lane * 16, xsrc + static_cast<int64_t>(8 * i) * d + k0);
#pragma unroll
            for (int i = 0; i < (RT::CE * (kKC / 4)) / 256; ++i)
                cp_async16(sw + (wr + (256 / (kKC / 4)) * i) * (kKC * 4) + wq * 16,
                           wsrc + static_cast<int64_t>((256 / (kKC / 4)) * i) * d + k0);
            return;
        }
        const int xpr = kc / 8;  // 16-byte pieces per x row
        for (int p = tid; p < RT::CT * xpr; p += 256) {
            const int r = p / xpr, q = p - (p / xpr) * xpr;
            const int t = min(ct0 + r, T - 1);
            cp_async16(sx + r * RT::XROW + q * 16, x + static_cast<int64_t>(t) * d + k0 + q * 8);
        }
        const int wpr = kc / 4;  // 16-byte pieces per Wg row
        for (int p = tid; p < RT::CE * wpr; p += 256) {
            const int r = p / wpr, q = p - (p / wpr) * wpr;
            const int e = min(ce0 + r, E - 1);
            cp_async16(sw + r * (kKC * 4) + q * 16, wg + static_cast<int64_t>(e) * d + k0 + q * 4);
        }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nk) load_stage(s, s * kKC);
        cp_async_commit();
    }

    float2 acc[kHP];  // pair p = a * 8 + b: token 2a + half, expert b; (.x, .y) = classes 2c, 2c+1
#pragma unroll
    for (int p = 0; p < kHP; ++p) acc[p] = make_float2(0.0f, 0.0f);

    for (int kc = 0; kc < nk; ++kc) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        {
            const int nxt = kc + kStages - 1;
            if (nxt < nk) load_stage(nxt % kStages, nxt * kKC);
            cp_async_commit();
        }
        const uint8_t* base = smem + (kc % kStages) * RT::SB;
        // this lane's 32-bit word (columns 2c, 2c+1) of token 2a + half of the warp's tile
        const uint32_t* sx = reinterpret_cast<const uint32_t*>(base + (wt * kTT + half) * RT::XROW) + c;
        const float2* sw = reinterpret_cast<const float2*>(base + RT::XB + (we * kTE) * (kKC * 4)) + c;
        const int steps = min(kKC, d - kc * kKC) / 32;
        // Operands of step s+1 are read from shared memory and widened to fp32
        // while the FMAs of step s run (two register sets, used in turn).
        float2 xa[HT], wa[kTE], xb[HT], wb[kTE];
        auto load_ops = [&](int s, float2(&xo)[HT], float2(&wo)[kTE]) {
#pragma unroll
            for (int a = 0; a < HT; ++a) {
                const uint32_t v = sx[(2 * a) * (RT::XROW / 4) + 16 * s];
                xo[a] = make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
            }
#pragma unroll
            for (int b = 0; b < kTE; ++b) wo[b] = sw[b * (kKC / 2) + 16 * s];
        };
        auto fma_step = [&](const float2(&xo)[HT], const float2(&wo)[kTE]) {
#pragma unroll
            for (int a = 0; a < HT; ++a)
#pragma unroll
                for (int b = 0; b < kTE; ++b) acc[a * kTE + b] = __ffma2_rn(xo[a], wo[b], acc[a * kTE + b]);
        };
        if (steps == kKC / 32) {  // full chunk: 8 steps, no guards
            load_ops(0, xa, wa);
#pragma unroll
            for (int s2 = 0; s2 < kKC / 64; ++s2) {
                load_ops(2 * s2 + 1, xb, wb);
                fma_step(xa, wa);
                if (2 * s2 + 2 < kKC / 32) load_ops(2 * s2 + 2, xa, wa);
                fma_step(xb, wb);
            }
        } else {  // last, partial chunk (d not a multiple of 256)
            for (int s = 0; s < steps; ++s) {
                load_ops(s, xa, wa);
                fma_step(xa, wa);
            }
        }
    }
    cp_async_wait<0>();

    // The fixed tree s_j += s_{j+off}, off = 16, 8, 4, 2 pairs class 2c+b with
    // class 2(c ^ 8)+b, 2(c ^ 4)+b, ... (the partner lane c ^ 8, ^ 4, ^ 2, ^ 1
    // of the same half); the last level, off = 1, adds the two classes a lane
    // holds.  After the four shuffle levels lane c holds pairs 4c .. 4c+3.
    reduce_level2<kHP / 2>(acc, c, 8);
    reduce_level2<kHP / 4>(acc, c, 4);
    reduce_level2<kHP / 8>(acc, c, 2);
    reduce_level2<kHP / 16>(acc, c, 1);
    constexpr int PPL = kHP / 16;  // pairs per lane after the reduction: PPL*c .. PPL*c + PPL-1
#pragma unroll
    for (int q = 0; q < PPL; ++q) {
        const int p = PPL * c + q;
        const int t = ct0 + wt * kTT + 2 * (p / kTE) + half;
        const int e = ce0 + we * kTE + (p % kTE);
        if (t < T && e < E) {
            float l = __fadd_rn(acc[q].x, acc[q].y);
            if (bias != nullptr) l = __fadd_rn(l, __ldg(bias + e));
            logits[static_cast<int64_t>(t) * E + e] = l;
        }
    }
}

}  // namespace route_detail
}  // namespace mk
