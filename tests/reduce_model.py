"""The summation tree of reduce_sum_f32, from the launch shape its header
states (include/sgemm_gb300.h: SGEMM_REDUCE_THREADS threads per block, at
most SGEMM_REDUCE_BLOCKS_PER_SM blocks per SM, four accumulators per thread
on 16-byte loads).  The GPU tests bound the kernel's error by
gamma_h * sum|x_i| (the oracle's ``sum_tolerance``) for the depth h computed
here; this module is test code and takes nothing from the product package.
"""

THREADS = 512          # SGEMM_REDUCE_THREADS
BLOCKS_PER_SM = 4      # SGEMM_REDUCE_BLOCKS_PER_SM


def blocks(n: int, num_sms: int) -> int:
    """Blocks of the launch: one per 16 * THREADS values, at most
    BLOCKS_PER_SM per SM, at least one."""
    return max(1, min(-(-n // (16 * THREADS)), BLOCKS_PER_SM * num_sms))


def tree_depth(n: int, num_sms: int, vec: bool) -> int:
    """Longest chain of FP32 additions any value goes through:
    a thread's own sequential adds into one accumulator (16-byte loads give
    each of the four accumulators one value per load, plus one for the
    n % 4 tail; 4-byte loads put every value into one accumulator), then
    (a0 + a1) + (a2 + a3) (2), the 32-lane shuffle tree (5), the combine of
    the block's 16 warp sums (5 levels of the same tree) and the blocks'
    atomic adds into *out, one after another (one per block)."""
    b = blocks(n, num_sms)
    g = b * THREADS
    if vec:
        chain = -(-(n // 4) // g) + (1 if n % 4 else 0)
    else:
        chain = -(-n // g)
    return chain + 2 + 5 + 5 + b
