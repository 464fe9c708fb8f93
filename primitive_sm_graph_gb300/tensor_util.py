"""dtype names shared by the binding and the graph builder (torch <-> psg)."""
import torch

_T2N = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16",
        torch.float64: "f64", torch.int32: "i32", torch.int16: "i16", torch.int8: "i8"}
_N2T = {v: k for k, v in _T2N.items()}


def dtype_name(dt: torch.dtype) -> str:
    try:
        return _T2N[dt]
    except KeyError:
        raise TypeError("dtype %s is not one of the seven" % dt) from None


def torch_dtype(name: str) -> torch.dtype:
    return _N2T[name]
