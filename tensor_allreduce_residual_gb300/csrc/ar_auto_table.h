// ar_auto_table.h -- measured choices for AR_AUTO on the fused path
// (the heuristic_min_warp_number / selectImplementation analogue of
// "allreduce.d2").
//
// Each entry covers one (element size, R, packed units per row) shape and the
// token counts up to `tokens_max`; the first matching entry wins.  `strategy`
// is AR_ONESHOT (1) or AR_TWOSHOT (2); `vpt` is the packed vectors each
// thread of the one-shot kernel keeps per row (threads per row =
// units_row / vpt rounded up to a power of two).  Shapes with no entry fall
// back to the rule in ar_api.cu.  The times in the comments are device time
// per call: replayed graphs below 64 MB of algorithmic bytes per call, and
// from 64 MB ("cold") back-to-back calls over input sets that together exceed
// L2 several times, so that every call reads its inputs from DRAM.
#pragma once

namespace ar {

struct AutoEntry {
    int esize;       // bytes per element
    int R;           // partials
    int units_row;   // 16-byte vectors per row
    int tokens_max;  // entry applies to tokens <= tokens_max
    int strategy;    // 1 = one-shot, 2 = two-shot
    int vpt;         // one-shot units per thread
    int mode;        // one-shot OneShotMode: 0 registers, 1 shared memory, 2 persistent, 3 bulk-copy ring
    int early;       // one-shot: 1 = write residual_out before the row barrier
    int blocks_per_sm = 1;  // one-shot mode 3: blocks per SM the grid is sized for
    int max_stages = 0;     // one-shot mode 3: ring slots per block at most (0: as many as fit)
};

static const AutoEntry kAutoTable[] = {
    {2, 2, 512, 1, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=1: one-shot 2.47 us
    {2, 2, 512, 2, 1, 1, 0, 0, 1, 0},  // tp_decode_R2_fp16_H4096 T=2: one-shot 2.352 us
    {2, 2, 512, 4, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=4: one-shot 2.349 us
    {2, 2, 512, 8, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=8: one-shot 2.406 us
    {2, 2, 512, 16, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=16: one-shot 2.381 us
    {2, 2, 512, 32, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=32: one-shot 2.39 us
    {2, 2, 512, 64, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=64: one-shot 2.48 us
    {2, 2, 512, 256, 1, 2, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=256: one-shot 3.005 us
    {2, 2, 512, 1024, 1, 2, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=1024: one-shot 6.128 us
    {2, 2, 512, 2147483647, 1, 1, 0, 1, 1, 0},  // tp_decode_R2_fp16_H4096 T=8192: one-shot 52.01 us cold
    {2, 2, 2048, 1, 1, 2, 4, 1, 8, 0},  // R2_bf16_H16384 T=1: one-shot 3.171 us
    {2, 2, 2048, 64, 1, 2, 4, 1, 4, 0},  // R2_bf16_H16384 T=64: one-shot 4.403 us
    {2, 2, 2048, 1024, 2, 0, 0, 0, 1, 0},  // R2_bf16_H16384 T=1024: two-shot 32.56 us cold
    {2, 2, 2048, 2147483647, 1, 4, 2, 1, 1, 0},  // R2_bf16_H16384 T=4096: one-shot 112.376 us cold
    {2, 3, 512, 1, 1, 1, 0, 1, 1, 0},  // R3_fp16_H4096 T=1: one-shot 2.918 us
    {2, 3, 512, 64, 1, 1, 0, 1, 1, 0},  // R3_fp16_H4096 T=64: one-shot 2.96 us
    {2, 3, 512, 2048, 1, 1, 3, 1, 2, 2},  // R3_fp16_H4096 T=2048: one-shot 18.012 us cold
    {2, 3, 512, 2147483647, 1, 1, 3, 1, 1, 4},  // R3_fp16_H4096 T=8192: one-shot 63.392 us cold
    {2, 4, 1024, 1, 1, 1, 4, 1, 8, 0},  // R4_fp16_H8192 T=1: one-shot 3.184 us
    {2, 4, 1024, 64, 1, 2, 0, 0, 1, 0},  // R4_fp16_H8192 T=64: one-shot 3.389 us
    {2, 4, 1024, 1024, 1, 4, 3, 0, 2, 0},  // R4_fp16_H8192 T=1024: one-shot 20.877 us cold
    {2, 4, 1024, 4096, 1, 4, 3, 1, 1, 4},  // R4_fp16_H8192 T=4096: one-shot 71.029 us cold
    {2, 4, 1024, 2147483647, 1, 4, 3, 1, 2, 2},  // R4_fp16_H8192 T=8192: one-shot 136.581 us cold
    {2, 8, 512, 1, 1, 1, 0, 1, 1, 0},  // R8_bf16_H4096 T=1: one-shot 2.909 us
    {2, 8, 512, 64, 1, 1, 0, 1, 1, 0},  // R8_bf16_H4096 T=64: one-shot 3.101 us
    {2, 8, 512, 1024, 1, 4, 1, 0, 1, 0},  // R8_bf16_H4096 T=1024: one-shot 16.744 us cold
    {2, 8, 512, 4096, 1, 1, 3, 1, 1, 2},  // R8_bf16_H4096 T=4096: one-shot 55.578 us cold
    {2, 8, 512, 2147483647, 1, 1, 3, 1, 1, 2},  // R8_bf16_H4096 T=8192: one-shot 106.717 us cold
    {2, 8, 1024, 1, 1, 1, 4, 1, 8, 0},  // R8_bf16_H8192 T=1: one-shot 3.206 us
    {2, 8, 1024, 8, 1, 1, 4, 1, 8, 0},  // R8_bf16_H8192 T=8: one-shot 3.315 us
    {2, 8, 1024, 32, 1, 1, 4, 1, 4, 0},  // R8_bf16_H8192 T=32: one-shot 3.83 us
    {2, 8, 1024, 64, 1, 2, 0, 1, 1, 0},  // R8_bf16_H8192 T=64: one-shot 4.019 us
    {2, 8, 1024, 256, 1, 2, 0, 1, 1, 0},  // R8_bf16_H8192 T=256: one-shot 5.789 us
    {2, 8, 1024, 512, 1, 4, 1, 0, 1, 0},  // R8_bf16_H8192 T=512: one-shot 17.295 us cold
    {2, 8, 1024, 1024, 1, 2, 3, 1, 1, 2},  // R8_bf16_H8192 T=1024: one-shot 29.86 us cold
    {2, 8, 1024, 2048, 1, 2, 3, 1, 1, 2},  // R8_bf16_H8192 T=2048: one-shot 56.376 us cold
    {2, 8, 1024, 4096, 1, 2, 3, 1, 1, 2},  // R8_bf16_H8192 T=4096: one-shot 106.507 us cold
    {2, 8, 1024, 2147483647, 1, 2, 3, 1, 1, 2},  // R8_bf16_H8192 T=8192: one-shot 207.824 us cold
    {2, 16, 1024, 1, 1, 1, 4, 1, 8, 0},  // R16_bf16_H8192 T=1: one-shot 4.934 us
    {2, 16, 1024, 64, 1, 1, 4, 1, 4, 0},  // R16_bf16_H8192 T=64: one-shot 5.642 us
    {2, 16, 1024, 2048, 1, 4, 3, 1, 1, 8},  // R16_bf16_H8192 T=2048: one-shot 97.094 us cold
    {2, 16, 1024, 2147483647, 1, 8, 3, 1, 1, 0},  // R16_bf16_H8192 T=8192: one-shot 365.917 us cold
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0},  // sentinel
};

// Measured choices for AR_AUTO on the reduce-only path (ar_sum, fusion
// NONE): which work partition was faster -- one slice over all blocks
// (strategy 1, the one-shot partition) or R rank slices (strategy 2, the
// two-shot reduce-scatter) -- per (element size, R), for n up to `units_max`
// 16-byte vectors (n / lanes).  Both partitions give bit-identical values,
// so the choice is speed only.  The first matching entry wins; an (element
// size, R) with no entry falls back to the rule in ar_api.cu.
struct SumAutoEntry {
    int esize;            // bytes per element
    int R;                // partials
    long long units_max;  // entry applies to nunits <= units_max
    int strategy;         // 1 = one slice, 2 = R rank slices
};

static const SumAutoEntry kSumAutoTable[] = {
    {2, 2, 2048LL, 2},  // 64..2048 vectors: 2 rank slices
    {2, 2, 524288LL, 1},  // 4096..524288 vectors: one slice
    {2, 2, 1048576LL, 2},  // 1048576..1048576 vectors: 2 rank slices
    {2, 2, 9223372036854775807LL, 1},  // 2097152..16777216 vectors: one slice
    {2, 3, 128LL, 1},  // 64..128 vectors: one slice
    {2, 3, 4096LL, 2},  // 256..4096 vectors: 3 rank slices
    {2, 3, 9223372036854775807LL, 1},  // 8192..16777216 vectors: one slice
    {2, 4, 64LL, 1},  // 64..64 vectors: one slice
    {2, 4, 2048LL, 2},  // 128..2048 vectors: 4 rank slices
    {2, 4, 262144LL, 1},  // 4096..262144 vectors: one slice
    {2, 4, 524288LL, 2},  // 524288..524288 vectors: 4 rank slices
    {2, 4, 9223372036854775807LL, 1},  // 1048576..16777216 vectors: one slice
    {2, 8, 128LL, 1},  // 64..128 vectors: one slice
    {2, 8, 2048LL, 2},  // 256..2048 vectors: 8 rank slices
    {2, 8, 32768LL, 1},  // 4096..32768 vectors: one slice
    {2, 8, 65536LL, 2},  // 65536..65536 vectors: 8 rank slices
    {2, 8, 9223372036854775807LL, 1},  // 131072..16777216 vectors: one slice
    {2, 16, 128LL, 1},  // 64..128 vectors: one slice
    {2, 16, 16384LL, 2},  // 256..16384 vectors: 16 rank slices
    {2, 16, 9223372036854775807LL, 1},  // 32768..16777216 vectors: one slice
    {4, 2, 128LL, 2},  // 128..128 vectors: 2 rank slices
    {4, 2, 256LL, 1},  // 256..256 vectors: one slice
    {4, 2, 2048LL, 2},  // 512..2048 vectors: 2 rank slices
    {4, 2, 16384LL, 1},  // 4096..16384 vectors: one slice
    {4, 2, 65536LL, 2},  // 32768..65536 vectors: 2 rank slices
    {4, 2, 131072LL, 1},  // 131072..131072 vectors: one slice
    {4, 2, 262144LL, 2},  // 262144..262144 vectors: 2 rank slices
    {4, 2, 524288LL, 1},  // 524288..524288 vectors: one slice
    {4, 2, 1048576LL, 2},  // 1048576..1048576 vectors: 2 rank slices
    {4, 2, 9223372036854775807LL, 1},  // 2097152..33554432 vectors: one slice
    {4, 3, 128LL, 1},  // 128..128 vectors: one slice
    {4, 3, 4096LL, 2},  // 256..4096 vectors: 3 rank slices
    {4, 3, 262144LL, 1},  // 8192..262144 vectors: one slice
    {4, 3, 524288LL, 2},  // 524288..524288 vectors: 3 rank slices
    {4, 3, 9223372036854775807LL, 1},  // 1048576..33554432 vectors: one slice
    {4, 4, 2048LL, 2},  // 128..2048 vectors: 4 rank slices
    {4, 4, 9223372036854775807LL, 1},  // 4096..33554432 vectors: one slice
    {4, 8, 2048LL, 2},  // 128..2048 vectors: 8 rank slices
    {4, 8, 65536LL, 1},  // 4096..65536 vectors: one slice
    {4, 8, 131072LL, 2},  // 131072..131072 vectors: 8 rank slices
    {4, 8, 524288LL, 1},  // 262144..524288 vectors: one slice
    {4, 8, 1048576LL, 2},  // 1048576..1048576 vectors: 8 rank slices
    {4, 8, 9223372036854775807LL, 1},  // 2097152..33554432 vectors: one slice
    {4, 16, 256LL, 1},  // 128..256 vectors: one slice
    {4, 16, 8192LL, 2},  // 512..8192 vectors: 16 rank slices
    {4, 16, 9223372036854775807LL, 1},  // 16384..33554432 vectors: one slice
    {0, 0, 0, 0},  // sentinel
};

}  // namespace ar
