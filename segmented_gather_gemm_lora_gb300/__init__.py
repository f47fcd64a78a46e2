"""GB300-native multi-adapter LoRA path (segmented gather GEMM, SGMV / BGMV).

The compute lives in liblora_sgmv.so (CUDA kernels for sm_103a behind the C ABI
declared in include/lora_sgmv.h); ``binding`` marshals torch tensors into it;
``workloads`` draws seeded synthetic inputs.
"""

__all__ = ["binding", "workloads", "build"]
