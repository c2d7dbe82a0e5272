"""Helpers shared by the GPU parity tests: moving seeded host arrays to the
device and wrapping oracle-quantized operands for the library's binding."""

import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def u8_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev())


def i32_to_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev())


def oracle_operand_rowwise(bits: np.ndarray, elem: str):
    """Oracle quantization of a K-major operand -> (binding operand on the
    device, dequantized float64 matrix)."""
    import fp8_bf16_mxfp4_gb300 as mxg
    data, scale = oracle.quantize_mx_rowwise(bits, elem)
    codes = oracle.unpack_e2m1(data) if elem == "e2m1" else data
    deq = oracle.dequantize_mx(codes, scale, elem)
    return mxg.MXOperand(u8_to_dev(data), u8_to_dev(scale), elem, bits.shape[1]), deq


def oracle_operand_colwise(bits: np.ndarray, splits, pad: int, elem: str, capacity: int | None = None):
    """Oracle column-wise segment-padded operand placed in a buffer of
    `capacity` columns (slack filled with arbitrary finite codes so that the
    GPU never relies on it being zero) -> (operand, dequantized [C, Spad],
    pad offsets)."""
    import fp8_bf16_mxfp4_gb300 as mxg
    data, scale, poff = oracle.quantize_mx_colwise_segment_padded(bits, splits, pad, elem)
    codes = oracle.unpack_e2m1(data) if elem == "e2m1" else data
    deq = oracle.dequantize_mx(codes, scale, elem)
    C, spad = codes.shape
    cap = capacity if capacity is not None else spad
    rng = np.random.default_rng(99)
    full = rng.integers(0, 0x7F, size=(C, cap)).astype(np.uint8)    # finite junk codes
    if elem == "e2m1":
        full &= 0x0F
    full[:, :spad] = codes
    fscale = rng.integers(100, 140, size=(C, cap // 32)).astype(np.uint8)
    fscale[:, : spad // 32] = scale
    fdata = oracle.pack_e2m1(full) if elem == "e2m1" else full
    return mxg.MXOperand(u8_to_dev(fdata), u8_to_dev(fscale), elem, cap), deq, poff
