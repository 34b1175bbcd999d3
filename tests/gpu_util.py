"""Moving seeded numpy operands to and from CUDA tensors (tests only)."""
import numpy as np


def dev(a, device="cuda", f16=False):
    """numpy fp32 array, or uint16 bit array of bf16 (or of fp16 when f16) ->
    CUDA tensor."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.float16 if f16 else torch.bfloat16)
    return torch.from_numpy(a).to(device)


def host_bits(t):
    """CUDA tensor -> numpy array of its raw bits (uint16/uint32/uint64)."""
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype == torch.float64:
        return t.view(torch.int64).numpy().view(np.uint64)
    raise TypeError(t.dtype)


def bits(a):
    """numpy array -> raw-bit view."""
    a = np.ascontiguousarray(a)
    return a.view({2: np.uint16, 4: np.uint32, 8: np.uint64}[a.dtype.itemsize])


def torch_dtype(dtype):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
