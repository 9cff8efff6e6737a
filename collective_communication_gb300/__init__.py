"""Ring AllReduce over N virtual ranks on one GB300 (sm_103a CUDA kernels
behind a C ABI), plus the one-shot AllReduce variant.

The Python layer only marshals arguments for the C ABI (librar.so, declared in
include/rar.h); every step of the collective runs in the CUDA kernels. Torch is
used for device memory and streams only. The binding is imported on first use
so that `collective_communication_gb300.inputs` stays importable without it.
"""
_BINDING_NAMES = (
    "RarError", "Status", "Dtype", "Proto", "load_library", "library_path", "allreduce", "oneshot",
    "workspace_bytes", "Workspace", "get_status", "strerror",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
