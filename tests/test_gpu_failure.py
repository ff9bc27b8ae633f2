"""The failure path on the GPU, made on purpose without a fault: a bounded
wait that runs out.

pa_test_expire_next_wait() makes the next multi-query launch skip the K loads
of each CTA's first key tile.  The MMA warp's wait for that tile is bounded
(about one second of GPU time): it must give up, set the library's device
error word, let the kernel drain and return -- no trap, no hang, the context
stays usable -- and the next call must be normal again.
"""
import pytest
import torch

from harness import DeviceWorkload, check_step
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_expired_wait_sets_the_error_word_and_the_next_call_is_clean():
    w = wl.random_small(501, dtype=wl.BF16, num_seqs=3, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=16, max_prior=200, max_q=30)
    assert pa.pa_device_error() == 0
    dw = DeviceWorkload(w)
    dw.scatter()
    pa.pa_test_expire_next_wait()
    dw.attention()                      # launches; the kernel gives up on one wait
    torch.cuda.synchronize()            # returns: no fault, no hang
    code = pa.pa_device_error()         # read and clear
    assert code != 0
    assert pa.pa_device_error() == 0    # cleared
    check_step(w)                       # the next call: parity, error word 0
