"""The all-reduce across the GPUs of one node (ar_comm_* and ar_allreduce_peer), on the one GPU here.

With one rank the sum over the ranks is the rank's own input, so out must equal
the input bit for bit, and the oracle's one-partial sum; the run still goes
through the whole kernel: the copy into the registered buffer, the block
barriers (each block signalling and awaiting itself), the rank-order sum, and
for two-shot the write-back and the gather.  Successive calls alternate the
two data areas and advance the epochs.

The bounded waits are tested in a child process on the test build: rank 0 of a
two-rank communicator over two local buffers, whose rank 1 never runs, so
rank 0's barrier waits on flags that nothing sets, run out after about a
second, and are reported by ar_device_status; the context stays usable.
Nothing here runs two ranks that wait on each other.
"""
import os
import subprocess
import sys

import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tensor_allreduce_residual_gb300 import _build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available()
    _build.build()
    ar.lib()


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("strategy", ["ONESHOT", "TWOSHOT", "AUTO"])
def test_one_rank_returns_its_input(dtype, strategy):
    comm = ar.PeerComm(0, 1, max_bytes=(1 << 22) * 4)
    for k, n in enumerate([1, 7, 8, 4097, 65536, (1 << 20) + 3, 1 << 22]):
        x = workloads.draw(("N", 0.0, 1.0), n, dtype, seed=k, k=0)
        got = comm.allreduce(x.cuda(), strategy=strategy)
        torch.cuda.synchronize()
        ref = oracle.sum([x], dtype)
        assert torch.equal(got.cpu().view(torch.uint8), ref.view(torch.uint8)), (dtype, strategy, n)
        assert torch.equal(got.cpu().view(torch.uint8), x.view(torch.uint8))
    assert ar.ar_device_status() == ar.AR_OK
    comm.close()


def test_one_rank_in_place_and_many_calls():
    comm = ar.PeerComm(0, 1, max_bytes=1 << 20)
    for call in range(7):   # both data areas, several epochs
        x = workloads.draw(("U", -1.0, 1.0), 100_003, "bf16", seed=call, k=1).cuda()
        keep = x.clone()
        comm.allreduce(x, out=x, strategy="TWOSHOT" if call % 2 else "ONESHOT")
        torch.cuda.synchronize()
        assert torch.equal(x.view(torch.int16), keep.view(torch.int16))
    assert ar.ar_device_status() == ar.AR_OK
    comm.close()


def test_errors_raise():
    comm = ar.PeerComm(0, 1, max_bytes=1024)
    with pytest.raises(ar.ARError) as e:
        comm.allreduce(torch.zeros(1024, dtype=torch.float32, device="cuda"))   # 4 KB > max_bytes
    assert e.value.status == ar.AR_ERR_WORKSPACE
    x = torch.zeros(100, dtype=torch.float16, device="cuda")
    with pytest.raises(ar.ARError) as e:
        comm.allreduce(x[1:])                                                   # misaligned
    assert e.value.status == ar.AR_ERR_UNSUPPORTED
    comm.close()
    with pytest.raises(RuntimeError):
        comm.allreduce(x)


def test_barrier_waits_run_out_when_a_rank_never_arrives():
    res = subprocess.run([sys.executable, "-m", "tests.peer_timeout_child"], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0 and "peer timeout ok" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]
