/*
 * devscan measurement hook -- not part of the product interface in
 * devscan.h.  Tests and benchmarks use it to run one operation through each
 * of its inter-block carry paths, so that every path is checked against the
 * oracle and timed against the others.  Production callers have no reason
 * to include this header: the default path is the one chosen by
 * measurement.
 *
 * P1 = geek-doc.cn/chip-design/intermediate/parallel-prefix-scan, "并行前缀和
 * scan: Hillis-Steele、Blelloch 与 warp shuffle 三种写法".
 */
#ifndef DEVSCAN_MEASURE_H
#define DEVSCAN_MEASURE_H

#include "devscan.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Inter-block carry strategy of the scans and their consumers (P1 section
 * 四 describes the three-phase "reduce, scan the block totals, add the
 * offsets" scheme and mentions chaining blocks inside one launch).  The
 * setting belongs to the CALLING THREAD: it changes the path of the devscan
 * calls that this thread makes afterwards and of no other thread's calls
 * (each thread starts on 0).  Modes:
 *   0 = default: scans of n <= 2^16 run in one thread-block cluster (up
 *       to 8 blocks exchanging their totals through distributed shared
 *       memory, any alignment); for 16-byte-aligned in/out the scans take 4
 *       for 2^17 <= n <= 2^24 and 3 above; compaction with flags takes 3 from
 *       n = 2^19 and 4 from 2^23; split_bit_u32 takes 4 from 2^20; the
 *       sorts' splits, the bracket scan and the segmented scan take 3 from
 *       n = 2^19; the bracket check without the scanned array (out == NULL)
 *       takes 4 from n = 2^17 (below 2^31); everything else takes 1;
 *   1 = one tile per block, single-pass decoupled look-back;
 *   2 = reduce-then-scan (three launches, one extra read of the input);
 *   3 = pipelined single pass: persistent warp-specialised blocks with bulk
 *       copies and a two-level look-back (16-byte-aligned in/out; others
 *       use 1);
 *   4 = L2-resident scan: one cooperative launch of one block per SM, a
 *       grid barrier between the chunk totals and the chunk scans, the
 *       second read served by L2 (16-byte-aligned in/out; others use 1;
 *       the fused-predicate compaction, split, the segmented scan and the
 *       bracket scan with its array stored use 3); the bracket check alone
 *       takes its one-read cooperative kernel at every size below 2^31, and
 *       compaction with flags and split_bit_u32 their two-launch paths (a
 *       count of 512-element parts with offsets per chunk of parts and
 *       carries between chunks, then a warp per part writing its runs).
 * Compaction and the split follow the same choice between 1 and 3 (their
 * pipelined kernels need 16-byte-aligned inputs, and flags too for
 * compaction).  Returns DEVSCAN_ERR_INVALID for any other mode (the
 * thread's setting is then unchanged). */
devscan_status devscan_measure_set_carry_mode(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DEVSCAN_MEASURE_H */
