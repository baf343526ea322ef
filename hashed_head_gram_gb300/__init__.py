"""GB300-native hashed multi-head N-gram memory lookup.

    hashed_head_gram_gb300.pg         the C-ABI binding (needs the built libpg.so)
    hashed_head_gram_gb300.workloads  seeded synthetic workloads (no lookup arithmetic)
    hashed_head_gram_gb300.build      builds libpg.so for sm_103a
"""
