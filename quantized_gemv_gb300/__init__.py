"""GB300-native batch-1 decode megakernel for Qwen3-0.6B-shaped transformers.

Submodules:
  mk        -- ctypes binding of the C-ABI library libmk.so (the product path)
  build     -- compiles libmk.so for sm_103a
  synthetic -- seeded synthetic inputs (weights, prompts, prefilled KV); no model arithmetic
Importing the package itself loads nothing; `quantized_gemv_gb300.mk` loads the CUDA library.
"""
