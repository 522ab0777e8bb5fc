"""Child process for test_peer_gpu: rank 0 of a two-rank communicator over two
local buffers (the test build's ar_comm_create_local), whose rank 1 never runs.
Every block barrier of rank 0's call waits for flags that nothing sets; the
waits must run out after about a second, the call must finish, ar_device_status
must report the timeout, and the context must stay usable."""
import ctypes
import sys
import time

import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads

ar.use_test_library()   # ar_comm_create_local exists in the test build only


def main():
    torch.cuda.set_device(0)
    L = ar.lib()
    assert ar.ar_device_status() == ar.AR_OK
    max_bytes = 1 << 20
    size = ar.ar_comm_buffer_size(2, max_bytes)
    bufs = [torch.empty(size, dtype=torch.uint8, device="cuda") for _ in range(2)]
    ptrs = (ctypes.c_void_p * 2)(*[b.data_ptr() for b in bufs])
    comm = ctypes.c_void_p(0)
    assert L.ar_comm_create_local(0, 2, ptrs, size, max_bytes, ctypes.byref(comm)) == ar.AR_OK
    x = torch.ones(4096, dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    torch.cuda.synchronize()
    t0 = time.time()
    assert L.ar_allreduce_peer(comm, x.data_ptr(), out.data_ptr(), x.numel(), ar.AR_FP16, ar.AR_ONESHOT, None) == 0
    torch.cuda.synchronize()
    took = time.time() - t0
    assert ar.ar_device_status() == ar.AR_ERR_TIMEOUT
    assert ar.ar_device_status() == ar.AR_OK           # the record was cleared
    assert 0.5 < took < 30.0, took
    assert L.ar_comm_destroy(comm) == ar.AR_OK
    # The context still works.
    s = workloads.reduce_only(4099, seed=3)
    got = ar.ar_sum([p.cuda() for p in s.partials])
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.int16), oracle.sum(s.partials, "fp16").view(torch.int16))
    assert ar.ar_device_status() == ar.AR_OK
    print(f"peer timeout ok ({took:.2f} s)")


if __name__ == "__main__":
    sys.exit(main())
