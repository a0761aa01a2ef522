// skv_ops.h -- operation count of the SKV v1 format's arithmetic, per scalar.
//
// The arithmetic roofline of the coder divides the format's own work by the
// rate at which this GPU executes that work. The work is counted here once,
// by instruction class, for one scalar of each of the four coding directions,
// following the format step by step (SKV v1 format, section 9 "Operation
// count", which prints the same table with the step each entry comes from):
// one C(o) of section 5 twice, the rANS step of section 6, the per-element
// inputs of section 4 and the word placement of section 7. The decoder's
// search for the code (beyond the two edges that bracket it) is not work of
// the format and is not counted. HBM traffic (the 16-byte KV, mu and output
// vectors, the bitstream words) is the byte roofline's and not counted here.
//
// skv_peak.cu runs one probe per class and one probe per table that issues
// exactly these counts per "scalar" with full instruction-level parallelism;
// the latter's scalars per second is the arithmetic roofline.
#pragma once

#include <cstdint>

namespace skv {

enum OpClass : int {
    kOpFp32 = 0,    // add / mul / fma .rn.f32
    kOpFminmax,     // min / max .f32
    kOpIadd,        // add / sub .u32 (a 64-bit add counts two)
    kOpLogic,       // and / or / xor / lop3, setp, selp, register moves of a 64-bit shift
    kOpShift,       // shl / shr / shf
    kOpIminmax,     // min / max .s32
    kOpImad,        // mul.lo / mad.lo .u32
    kOpImadHi,      // mul.hi / mad.hi .u32
    kOpImadWide,    // mul.wide.u32 (32 x 32 -> 64 bits: two 32-bit results)
    kOpCvt,         // conversions between binary32 and integers
    kOpMufu,        // rcp / lg2 / ex2 .approx
    kOpPopc,        // popc
    kOpVote,        // vote.ballot
    kOpLds,         // shared-memory load
    kOpLdt,         // load from a small global table (L1-resident)
    kOpSts,         // shared-memory store
    kNumOpClasses
};

// 32-bit operations per instruction of each class.
constexpr uint32_t kOpWeight[kNumOpClasses] = {1, 1, 1, 1, 1, 1, 1, 1, 2, 1, 1, 1, 1, 1, 1, 1};

enum OpTable : int { kTabBf16Encode = 0, kTabBf16Decode, kTabE4m3Encode, kTabE4m3Decode, kNumOpTables };

// Per-scalar instruction counts, classes in OpClass order:
//            fp32 fmnx iadd logic shift imnx imad hi wide cvt mufu popc vote lds ldt sts
constexpr uint32_t kOpCount[kNumOpTables][kNumOpClasses] = {
    /* bf16 encode */ {8, 4, 21, 16, 18, 4, 12, 4, 3, 7, 1, 1, 1, 4, 3, 1},
    /* bf16 decode */ {6, 4, 16, 16, 17, 4, 11, 4, 3, 2, 0, 2, 1, 5, 3, 0},
    /* e4m3 encode */ {8, 4, 21, 16, 17, 4, 12, 4, 3, 7, 1, 1, 1, 9, 1, 1},
    /* e4m3 decode */ {6, 4, 16, 16, 16, 4, 11, 4, 3, 2, 0, 2, 1, 10, 1, 0},
};

constexpr uint32_t op_instructions(int t) {
    uint32_t n = 0;
    for (int c = 0; c < kNumOpClasses; ++c) n += kOpCount[t][c];
    return n;
}
constexpr uint32_t op_weighted(int t) {
    uint32_t n = 0;
    for (int c = 0; c < kNumOpClasses; ++c) n += kOpCount[t][c] * kOpWeight[c];
    return n;
}

}  // namespace skv
