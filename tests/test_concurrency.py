"""Calls from several host threads at once (the C ABI promises reentrant calls from any host thread).

Every thread runs its own stream and its own mix of entry points: the device forward (unsplit and
with split keys, whose workspace is taken stream-ordered inside the call), the forward on host
buffers (whose copy streams are shared per device and guarded by a lock), the backward and the
split-KV decode.  The kernels are deterministic, so each result must equal, bit for bit, the same
call made alone on the default stream.
"""
import threading

import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu


def _jobs(dev, tid):
    """The calls of thread `tid`: a list of (name, callable(stream) -> tuple of tensors)."""
    d = 64 if tid % 2 == 0 else 128
    q, k, v = make_qkv(1, 2 + tid, 300 + 37 * tid, 700 + 91 * tid, d, "bf16", seed=4100 + tid, device=dev)
    qs, ks, vs = make_qkv(1, 1, 1000, 3000, 64, "bf16", seed=4200 + tid, device=dev)
    qd, kd, vd = make_qkv(2, 4, 1, 5000 + 13 * tid, 64, "bf16", seed=4300 + tid, device=dev)
    dout = make_dout(1, 2 + tid, 300 + 37 * tid, d, "bf16", seed=4400 + tid, device=dev)
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))

    def fwd(s):
        return fa.fa_fwd(q, k, v, stream=s, causal=bool(tid & 1))

    def fwd_split(s):
        return fa.fa_fwd(qs, ks, vs, stream=s, kv_splits=4)

    def fwd_host(s):
        o, lse = fa.fa_fwd_host(hq, hk, hv, stream=s)
        s.synchronize()  # host results are valid once the stream has finished
        return o.clone(), lse.clone()

    def bwd(s):
        o, lse = fa.fa_fwd(q, k, v, stream=s)
        return fa.fa_bwd(q, k, v, o, dout, lse, stream=s)

    def decode(s):
        return fa.fa_decode_splitkv_ex(qd, kd, vd, 7, with_lse=True, stream=s)

    return [("fwd", fwd), ("fwd_split", fwd_split), ("fwd_host", fwd_host), ("bwd", bwd), ("decode", decode)]


def _as_tuple(r):
    return tuple(x for x in (r if isinstance(r, tuple) else (r,)) if x is not None)


def test_calls_from_four_host_threads(cuda_device):
    n_threads, rounds = 4, 3
    jobs = [_jobs(cuda_device, t) for t in range(n_threads)]
    # each call alone, on the default stream
    ref = []
    for tj in jobs:
        s = torch.cuda.current_stream()
        ref.append([tuple(x.clone() for x in _as_tuple(fn(s))) for _, fn in tj])
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK

    results = [[] for _ in range(n_threads)]
    errors = []
    start = threading.Barrier(n_threads)

    def run(tid):
        try:
            torch.cuda.set_device(cuda_device)
            s = torch.cuda.Stream(device=cuda_device)
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(rounds):
                    for name, fn in jobs[tid]:
                        results[tid].append((name, tuple(x.clone() for x in _as_tuple(fn(s)))))
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=run, args=(t,)) for t in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
        assert not t.is_alive(), "a host thread did not finish"
    torch.cuda.synchronize()
    assert not errors, errors
    assert fa.fa_check_device_error() == fa.FA_OK
    for tid in range(n_threads):
        assert len(results[tid]) == rounds * len(jobs[tid])
        for i, (name, got) in enumerate(results[tid]):
            want = ref[tid][i % len(jobs[tid])]
            assert len(got) == len(want), (tid, name)
            for g, w in zip(got, want):
                assert torch.equal(g.cpu(), w.cpu()), f"thread {tid}, {name}: differs from the call made alone"
