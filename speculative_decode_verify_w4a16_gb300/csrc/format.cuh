// Packed ("streaming") layout of the int4 g128 weights, shared by the
// prepack kernel and the linear kernels.
//
// The matrix is cut into units of 128 rows x 128 K (one quantisation group
// of 128 rows); units are stored in (row-tile t, group g) order, unit index
// u = t * G + g with G = K / 128, so a row-tile's K range is contiguous and a
// CTA can stream any contiguous range of units with 1-D bulk copies.
//
// Inside a unit (8192 bytes = 2048 uint32):
//   word = (((w4 * 2 + rt) * 2 + h) * 32 + lane) * 4 + j
//     w4   0..3  32-row slice (rows 32*w4 ..) — one consumer warp, and one
//                TMEM lane quadrant on the tensor-memory path
//     rt   0..1  16-row tile inside the slice: r0 = 32*w4 + 16*rt
//     h    0..1  K half (k 0..63 / 64..127 of the group)
//     lane 0..31 lane = 4*gid + c (gid 0..7, c 0..3)
//     j    0..3  16-wide K step inside the half: kb = 16*(4*h + j)
//   nibble positions of that word (codes stored offset-binary, code + 8):
//     bits  0: (r0+gid,   kb+4c)     bits 16: (r0+gid,   kb+4c+1)
//     bits  4: (r0+gid+8, kb+4c)     bits 20: (r0+gid+8, kb+4c+1)
//     bits  8: (r0+gid,   kb+4c+2)   bits 24: (r0+gid,   kb+4c+3)
//     bits 12: (r0+gid+8, kb+4c+2)   bits 28: (r0+gid+8, kb+4c+3)
// so (word >> 4i) & 0x000F000F yields, for i = 0..3, the bf16x2 pairs
//   (row gid, k 4c..4c+1), (row gid+8, k 4c..4c+1),
//   (row gid, k 4c+2..4c+3), (row gid+8, k 4c+2..4c+3)
// i.e. one m16n8k16 A fragment (with the K order inside each 16-step
// permuted the same way for A and B) and one 16x256b TMEM fragment.
//
// Scales of a unit (128 halves = 256 bytes): half = ((w4 * 8 + gid) * 2 + rt) * 2 + hi
// for row 32*w4 + 16*rt + gid + 8*hi, so a lane reads its four scales as one
// 8-byte load.
#pragma once

#include <stdint.h>

namespace w4a16 {

constexpr int kUnitRows = 128;
constexpr int kGroup = 128;
constexpr int kUnitWords = 2048;       // uint32 per unit
constexpr int kUnitBytes = 8192;
constexpr int kUnitScaleBytes = 256;

}  // namespace w4a16
