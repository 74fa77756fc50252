"""The Python binding's own checks, which run before any CUDA call: tensors
that are not 2-D (3-D for bmm) float32 CUDA tensors and mismatched shapes
raise SgemmError with status -1, so nothing reaches the library."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding


def _raises(fn, *args, match, **kw):
    with pytest.raises(binding.SgemmError) as err:
        fn(*args, **kw)
    assert err.value.status == -1 and match in str(err.value), str(err.value)


def test_sgemm_rejects_host_and_non_float32_tensors():
    A, B, C = torch.zeros(4, 3), torch.zeros(3, 5), torch.zeros(4, 5)
    _raises(binding.sgemm, A, B, C, match="A must be a 2-D float32 CUDA tensor")
    _raises(binding.sgemm_ex, A.double(), B, C, match="A must be a 2-D float32 CUDA tensor")
    _raises(binding.matmul, A, B, C, match="must be a 2-D float32 CUDA tensor")


def test_sgemm_rejects_mismatched_shapes():
    _raises(binding.sgemm_ex, torch.zeros(4, 3), torch.zeros(2, 5), torch.zeros(4, 5), match="shape mismatch")
    _raises(binding.sgemm_ex, torch.zeros(4, 3), torch.zeros(3, 5), torch.zeros(5, 4), match="shape mismatch")


def test_bmm_checks():
    _raises(binding.bmm, torch.zeros(4, 3), torch.zeros(3, 5), torch.zeros(4, 5), match="bmm takes 3-D tensors")
    _raises(binding.bmm, torch.zeros(2, 4, 3), torch.zeros(3, 3, 5), torch.zeros(2, 4, 5), match="shape mismatch")
    _raises(binding.bmm, torch.zeros(2, 4, 3), torch.zeros(2, 3, 5), torch.zeros(2, 4, 5),
            match="must be a 2-D float32 CUDA tensor")


def test_reduce_sum_rejects_host_tensors():
    _raises(binding.reduce_sum, torch.zeros(100), match="x must be a contiguous float32 CUDA tensor")
