"""Concurrent use of the library: GEMMs from two host threads on their own
streams (tensor-map caches are per thread, options and device state shared),
interleaved launches on two streams from one thread, and host-operand GEMMs
from two threads (the copy streams inside the library are shared)."""
import threading

import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, run_gemm

pytestmark = pytest.mark.gpu


def test_two_threads_two_streams():
    cases = [("bf16", 1024, 1536, 512, 61), ("nvfp4", 768, 1024, 1024, 62)]
    prepared = []
    for fmt, m, n, k, seed in cases:
        ops = Operands(fmt, m, n, k, seed)
        prepared.append((fmt, m, n, k, ops, ops.upload()))
    results, errors = {}, []

    def work(i):
        try:
            fmt, m, n, k, ops, dev = prepared[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = [run_gemm(fmt, dev, m, n, k, 1.0, stream=s.cuda_stream) for _ in range(20)]
            s.synchronize()
            results[i] = outs
        except Exception as e:   # surfaced in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(prepared))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert tkg.device_status() == tkg.OK
    for i, (fmt, m, n, k, ops, _) in enumerate(prepared):
        ref, S = ops.reference(rows=(0, 128))
        first = results[i][0]
        for D in results[i]:
            assert torch.equal(D.view(torch.int16), first.view(torch.int16))
        assert_within_tolerance(bf16_to_f64(first[:128]), ref, S, f"{fmt} from a second thread")


def test_interleaved_streams_one_thread():
    ops_a = Operands("mxfp8", 512, 768, 512, 63)
    ops_b = Operands("bf16", 300, 264, 320, 64)
    dev_a, dev_b = ops_a.upload(), ops_b.upload()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(10):
        outs.append(("a", run_gemm("mxfp8", dev_a, 512, 768, 512, 1.0, stream=s1.cuda_stream)))
        outs.append(("b", run_gemm("bf16", dev_b, 300, 264, 320, 1.0, stream=s2.cuda_stream)))
    torch.cuda.synchronize()
    assert tkg.device_status() == tkg.OK
    ref_a, S_a = ops_a.reference()
    ref_b, S_b = ops_b.reference()
    for tag, D in outs:
        ref, S = (ref_a, S_a) if tag == "a" else (ref_b, S_b)
        assert_within_tolerance(bf16_to_f64(D), ref, S, f"stream {tag}")


def test_from_host_two_threads():
    # each thread: its own pinned host operands, staging buffers and stream;
    # three calls each, enqueued while the other thread enqueues its own
    cases = [(4096, 2048, 512, 71), (2560, 4104, 256, 72)]
    prepared = []
    for m, n, k, seed in cases:
        ops = Operands("bf16", m, n, k, seed)
        Ah = torch.from_numpy(np.ascontiguousarray(ops.A).view(np.int16)).view(torch.bfloat16).pin_memory()
        Bh = torch.from_numpy(np.ascontiguousarray(ops.B).view(np.int16)).view(torch.bfloat16).pin_memory()
        dev = [torch.empty((m, k), dtype=torch.bfloat16, device="cuda"),
               torch.empty((n, k), dtype=torch.bfloat16, device="cuda"),
               torch.empty((m, n), dtype=torch.bfloat16, device="cuda")]
        outs = [torch.empty((m, n), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
        prepared.append((ops, Ah, Bh, dev, outs))
    errors = []

    def work(i):
        try:
            ops, Ah, Bh, dev, outs = prepared[i]
            s = torch.cuda.Stream()
            for Dh in outs:
                tkg.gemm_bf16_from_host(Ah, Bh, Dh, dev[0], dev[1], dev[2], stream=s)
            s.synchronize()
        except Exception as e:   # surfaced in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(prepared))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert tkg.device_status() == tkg.OK
    for ops, _, _, _, outs in prepared:
        ref, S = ops.reference(rows=(ops.m - 64, 64))
        for Dh in outs:
            assert torch.equal(Dh.view(torch.int16), outs[0].view(torch.int16))
        assert_within_tolerance(bf16_to_f64(outs[0])[ops.m - 64:], ref, S, f"from_host thread {ops.m}x{ops.n}")
