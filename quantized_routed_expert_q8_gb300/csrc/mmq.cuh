// Declarations shared by the grouped MMQ kernels and the C-ABI layer.
#pragma once

#include "common.cuh"

namespace moe {

// indices into the workspace counter array (uint32 counters[48])
enum { MMQ_COUNTER_NTILES = 0, MMQ_COUNTER_TICKET = 1 };

int launch_mmq_tiles(const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                     int E, int R, int BM, uint8_t* ws, const WsLayout& W, cudaStream_t stream);

// Optional fused epilogues of the MMQ; all null: plain h / y rows.  The
// folded-scale kernel takes the down projection's combine (comb), not the
// gate/up re-quantization (hq).
struct MmqFused {
    int8_t* hq = nullptr;      // gate/up: q8_1 hidden quants [R][f] written instead of h
    uint16_t* hds = nullptr;   // gate/up: (d, s) binary16 pairs [R][f/32]
    float* comb = nullptr;     // down: combined output [T][d], besides y
    const int32_t* src = nullptr;
    const int32_t* slot = nullptr;
    const float* w = nullptr;
    int32_t* arrivals = nullptr;  // [T][d/256], set by launch_combine_arrivals
    int K = 0, T = 0;
};

// The grouped MMQ with the block scales folded into binary16 hi + lo operands
// (stages 4 and 6 on the tensor cores; shapes with d % 256 == 0, f % 128 == 0).
bool mmq_fold_supported(int wtype, int d, int f);
int launch_mmq_fold(int wtype, bool gateup, const uint8_t* group_base, size_t slot_stride,
                    const int32_t* active, const int32_t* n_active, const int32_t* offsets, int E,
                    const int8_t* xq, const uint16_t* xds, int R, int d, int f, float* out,
                    uint8_t* ws, const WsLayout& W, const MmqFused& F, cudaStream_t stream);

int launch_combine_arrivals(const int32_t* slot, int T, int K, int R, int d, int32_t* arrivals,
                            float* out, cudaStream_t stream);

// SiLU(g) * u in fp32 with SiLU(g) = g / (1 + exp(-g)), IEEE division.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

}  // namespace moe
