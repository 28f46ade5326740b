"""precision_linear_gb300: the NVFP4 + LoRA + AQN-RMSNorm linear of quantised RL
rollout, as hand-written CUDA kernels for sm_103a behind a C ABI.

Public calls (thin ctypes marshalling in ``binding``; all arithmetic runs in
``libprecision_linear.so``):

* ``nvfp4_quantize(W)`` -> (codes, scales, s_g)
* ``rmsnorm_aqn(x, w_norm, z, eps)`` -> h
* ``nvfp4_lora_linear(x, codes, scales, s_g, A, B, lam, w_norm, z, eps)`` -> y

``synthetic`` holds the seeded workload generators and imports no native code.
The binding is loaded on first use of a public call and raises if the shared
library has not been built.
"""

_BINDING_NAMES = {
    "nvfp4_quantize", "rmsnorm_aqn", "nvfp4_lora_linear", "workspace_bytes",
    "nvfp4_bytes", "lib", "PLError", "Workspace",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
