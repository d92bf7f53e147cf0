"""Shared helpers of the GPU parity tests (inputs from synth, expectations from oracle)."""
import numpy as np
import torch

import oracle
import synth
import lossless_bit_weights_gb300 as w12


def to_dev16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def to_np16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def f32_of_bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def canonical_np(A):
    c = w12.w12_export_canonical(A)
    torch.cuda.synchronize()
    return dict(hi=c["hi"].cpu().numpy(), lo=c["lo"].cpu().numpy(), base=c["base"].cpu().numpy(),
                rowptr=c["rowptr"].cpu().numpy().view(np.uint32), esc=c["esc"].cpu().numpy().view(np.uint32))


def assert_canonical_equal(A, enc: "oracle.Encoded"):
    c = canonical_np(A)
    assert np.array_equal(c["base"], enc.base), "base"
    assert np.array_equal(c["hi"], enc.hi), "hi plane"
    assert np.array_equal(c["lo"], enc.lo), "lo plane"
    assert np.array_equal(c["rowptr"], enc.rowptr), "rowptr"
    assert np.array_equal(c["esc"], enc.esc), "escapes"
    assert A.n_esc == enc.n_esc


def assert_gemm_close(y_gpu: np.ndarray, y64: np.ndarray, B: np.ndarray, rel: float = 1e-4):
    """|y - y64| <= rel * sum|x*w| elementwise (the bound fp32 accumulation must meet)."""
    err = np.abs(y_gpu.astype(np.float64) - y64)
    bad = err > rel * B
    assert not bad.any(), f"{int(bad.sum())} outputs outside {rel}*B; worst ratio {(err / np.maximum(B, 1e-300)).max():.3g}"
    return float((err / np.maximum(B, 1e-300)).max())


def device_weights(seed, layer, tensor, N, K) -> torch.Tensor:
    W = torch.empty((N, K), dtype=torch.int16, device="cuda")
    synth.weights_dev(seed, layer, tensor, W)
    return W
