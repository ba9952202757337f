"""GB300-native paged speculative verification: paged_verify_attn, spec_accept,
spec_accept_tree and block_table_commit behind a C ABI (libsvpa.so).

``svpa`` is the ctypes binding (argument marshalling only); ``workloads`` draws
seeded synthetic inputs.
"""
