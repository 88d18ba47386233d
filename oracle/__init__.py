"""fp64 CPU oracle for query-aware sparse-page decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package
smoke check and the benchmark's CPU-baseline leg may import or run this.
It shares no code with the CUDA path: it is plain numpy, written step by
step from the pages, with no blocking, fusion or reordering beyond what a
step's definition states.

Modules
  quest     per-page per-channel min/max metadata and the Quest upper-bound
            page score (Quest 完全拆解, 核心机制 / 关键性估计算法)
  sketch    SALS-style index key: fixed Gaussian low-rank projection, int4
            per-block quantisation, group-mean int8 index query, integer dot,
            block log-sum-exp (SALS长序列推理优化, Quant Sals Indexer steps 1-5)
  select    exact top-k with forced sink/recent (or tail) pages, lower page
            index winning ties (SALS QSI Top-k 计算实现; Day 10·2 确定性红线)
  attention exact softmax attention over the gathered pages, fp64
            (SALS SFAA; Quest 三段式 kernel, Approximate attention)
  decode    one whole decode step built from the above
  bytes     the read-ratio / byte model (Quest 三段式 kernel 与内存流水)

Parity unpinned: whether the SALS reading (sketch.py) matches the real QSI
operator.  Its formulas were lost from the page's text, so it is pinned
only against the definition written here and the special cases tested
against it (identity projection without quantisation = exact block
log attention mass; brute-force integer dots; quantisation error bounds).
"""
