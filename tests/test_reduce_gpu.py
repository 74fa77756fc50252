"""GPU parity of reduce_sum_f32 against the FP64 sum oracle: within the
gamma_h bound of the summation tree of the launch shape the header states
(tests/reduce_model.py) on real values, exact on small integers (every
partial sum an integer below 2^24)."""
import numpy as np
import pytest
import torch

import oracle
import reduce_model
from dense_fp32_gemm_06_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def run(x_np, offset=0):
    buf = np.zeros(x_np.size + offset + 8, np.float32)
    buf[offset:offset + x_np.size] = x_np
    t = torch.from_numpy(buf).cuda()
    out = torch.full((1,), float("nan"), device="cuda")
    st = binding.reduce_sum_raw(t.data_ptr() + 4 * offset, x_np.size, out.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    return float(out.item())


@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 1023, 4099, (1 << 20) + 7, 1 << 24])
@pytest.mark.parametrize("offset", [0, 1])
def test_reduce_real_values(n, offset):
    x = inputs.draw_matrix("normal", n + offset, 0, 1, n)[0] if n else np.zeros(0, np.float32)
    got = run(x, offset)
    s, a = oracle.sum_f64(x)
    depth = reduce_model.tree_depth(n, torch.cuda.get_device_properties(0).multi_processor_count,
                                    vec=offset % 4 == 0)
    assert oracle.sum_within_tolerance(got, s, a, depth), (got, s, oracle.sum_tolerance(a, depth))


@pytest.mark.parametrize("n", [7, 100003, 1 << 21])
def test_reduce_integers_exact(n):
    x = inputs.draw_matrix("int", n, 0, 1, n)[0]
    assert run(x) == oracle.sum_f64(x)[0]


def test_reduce_full_size():
    """2^28 values (1 GiB), the bandwidth-bound size the measurement uses."""
    n = 1 << 28
    x = torch.empty(n, device="cuda").uniform_(-1, 1)
    got = binding.reduce_sum(x).item()
    xh = x.cpu().numpy()
    s, a = oracle.sum_f64(xh)
    depth = reduce_model.tree_depth(n, torch.cuda.get_device_properties(0).multi_processor_count, vec=True)
    assert oracle.sum_within_tolerance(got, s, a, depth)


def test_reduce_argument_checks():
    assert binding.reduce_sum_raw(0, 5, 256) == 1
    assert binding.reduce_sum_raw(258, 5, 256) == 1
    assert binding.reduce_sum_raw(256, -1, 256) == 2
    assert binding.reduce_sum_raw(256, 5, 0) == 3
