"""GB300 (sm_103a) paged multi-token KV attention.

``pkv`` is the Python binding of the C library (include/pkv.h): a KV block
pool, the paged KV append, generalised paged attention (several new query
tokens per request over a block-table-addressed cache, causal on absolute
position), and block swap to a CPU tier.  ``workloads`` draws seeded
synthetic batches; ``build`` compiles the library.  Importing the package
does not load the CUDA library; the first call into ``pkv`` does, and fails
loudly if it has not been built.
"""
