"""CPU oracle for the DCP sparse-indexer path.  TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy restatements of what each step of the path
computes, written from the pages that describe it (PR #46076 report "[Attention]
[DSA] support dcp for FLASHINFER_MLA_SPARSE"; PR #40996 report "DCP supports
hybrid attention").  Floating-point arithmetic that the pages leave open is done
in fp64.

Only the test suite, the package's smoke check and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it, and it shares no
code with the CUDA library: the only common module is `workloads`, which draws
seeded random inputs and holds none of the method's arithmetic.

Modules:
  dcp_layout  which shard holds a token, local positions, splitting a global
              logits row into per-shard rows (all by counting, from the rule)
  indexer     global top-K definition, shard top-K, candidate packing, stable
              merge, index conversion with compaction
  combine     LSE combine of per-shard partial attention outputs (fp64)
  pipeline    the steps chained for one workload
  attention   each shard's sparse MLA decode over its selected slots (fp64)
  kv_write    the write-side slot mapping of new tokens
  indexer_logits  the indexer's ReLU-weighted head sum of fp8 query-key dot
              products over each shard's paged key cache (fp64)
  pcp_prefill the PCP prefill cache rows: RMS norm of kv_c, interleaved
              rotation of k_pe, the ranks' gather, the cache insert (fp64)

Every function is pinned by a `-m "not gpu"` test against something other than
itself (brute force, a worked example on the pages, closed forms, invariants).
"""
