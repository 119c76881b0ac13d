"""libmla: paged MLA decode attention for sm_103a behind a C ABI.

``workloads`` (seeded synthetic inputs) imports without a GPU; the CUDA
binding lives in ``libmla`` and fails loudly when the compiled library is
missing.
"""
