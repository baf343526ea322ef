"""CPU oracle for the hashed multi-head N-gram lookup -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs
may import anything from here. The product library never does: it shares no code
with this package and fails loudly when its own CUDA build is missing.

  oracle/pg_oracle.c  plain C: canonical map, n-grams, hashes, row indices, sign
                      words, NF4 decode, signed concat / flat sum (bit-exact parts)
  oracle/oracle.py    ctypes wrapper + row fetch (numpy fancy indexing)
  oracle/dense.py     fp64 numpy: projection, scalar gate, RMSNorm-sigmoid gate,
                      causal depthwise conv + SiLU + residual
  oracle/nf4_levels.py  derivation of the 16 NF4 levels from normal quantiles
"""
