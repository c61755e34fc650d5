"""Runtime behaviour on the GPU: determinism, streams, the bounded-wait
timeout path, and that a call with bad arguments launches nothing."""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import Workload, make_inputs
from tests.gpu_helpers import Run, check, compare_full, to_device

pytestmark = pytest.mark.gpu


def test_bitwise_deterministic(cuda_lib):
    """Static schedule, no atomics: two calls give identical bits."""
    w = Workload("t", 2, 8, 1000, 1000, 128, "bf16", "BNSD", True, seed=21)
    x = make_inputs(w, device="cuda")
    a = Run(w, x.q, x.k, x.v)
    b = Run(w, x.q, x.k, x.v)
    torch.cuda.synchronize()
    assert a.status == 0 and b.status == 0
    assert torch.equal(a.o.view(torch.int16), b.o.view(torch.int16))
    assert torch.equal(a.lse.view(torch.int32), b.lse.view(torch.int32))


def test_side_stream(cuda_lib):
    w = Workload("t", 1, 4, 300, 300, 64, "f16", "BSND", False, seed=22)
    x = make_inputs(w)
    q, k, v = to_device(x)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        r = Run(w, q, k, v, stream=s.cuda_stream)
    s.synchronize()
    eo, el, og, lg = compare_full(w, r, x)
    check(w, r, eo, el, og, lg)


def test_wait_timeout_reports_and_context_survives(cuda_lib):
    """A wait on a barrier nothing arrives at must expire after its limit,
    report FA_ERR_DEVICE_TIMEOUT, and leave the context usable."""
    st = binding.fa_probe_wait_timeout(2_000_000)   # 2 ms limit
    assert st == 5, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0       # the word was cleared
    w = Workload("t", 1, 2, 256, 256, 128, "bf16", "BNSD", True, seed=23)
    x = make_inputs(w)
    q, k, v = to_device(x)
    r = Run(w, q, k, v)
    torch.cuda.synchronize()
    eo, el, og, lg = compare_full(w, r, x)
    check(w, r, eo, el, og, lg)


def test_bad_arguments_launch_nothing(cuda_lib):
    w = Workload("t", 1, 1, 128, 128, 128, "bf16", "BNSD", False, seed=24)
    x = make_inputs(w, device="cuda")
    o = torch.full_like(x.q, 7.0)
    lse = torch.full((1, 1, 128), 7.0, device="cuda")
    st = binding.fa_fwd(x.q.data_ptr(), x.k.data_ptr(), x.v.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), 1, 1, 128, 128, 96, 0.1, "BNSD", 0, "bf16")
    assert st == 2
    st = binding.fa_fwd(x.q.data_ptr() + 2, x.k.data_ptr(), x.v.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), 1, 1, 128, 128, 128, 0.1, "BNSD", 0, "bf16")
    assert st == 3
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())


def test_torch_tensor_wrapper(cuda_lib):
    w = Workload("t", 2, 2, 200, 300, 128, "bf16", "BSND", True, seed=25)
    x = make_inputs(w)
    q, k, v = to_device(x)
    out, lse = binding.attention(q, k, v, causal=True, layout="BSND")
    torch.cuda.synchronize()
    O, L = oracle.attention_full(x.q, x.k, x.v, dtype="bf16", layout="BSND", B=2, H=2, S_q=200,
                                 S_kv=300, D=128, scale=w.softmax_scale, causal=True)
    og = out.float().cpu().double().permute(0, 2, 1, 3).numpy()
    assert np.abs(og - O).max() <= 1.6e-2
    assert np.abs(lse.cpu().double().numpy() - L).max() <= 1e-3


def test_calls_from_a_thread_that_never_touched_the_device(cuda_lib):
    # The first CUDA call of a new thread is the library's own: it must make
    # the device's context current itself (tensor-map encoding needs one).
    import threading
    from tiled_attention_10_gb300.inputs import Workload, make_inputs
    w = Workload("t", 1, 2, 300, 300, 128, "bf16", "BNSD", True, seed=3)
    x = make_inputs(w, device="cuda")
    o1, o2 = torch.empty_like(x.q), torch.empty_like(x.q)
    l1, l2 = (torch.empty(1, 2, 300, device="cuda") for _ in range(2))
    args = lambda o, l: (x.q.data_ptr(), x.k.data_ptr(), x.v.data_ptr(), o.data_ptr(), l.data_ptr(),
                         1, 2, 300, 300, 128, w.softmax_scale, "BNSD", True, "bf16", None, None, None)
    assert binding.fa_fwd(*args(o1, l1)) == 0
    res = {}
    t = threading.Thread(target=lambda: res.setdefault("st", binding.fa_fwd(*args(o2, l2))))
    t.start()
    t.join()
    torch.cuda.synchronize()
    assert res["st"] == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.parametrize("split", [False, True])
def test_dependent_calls_back_to_back(split, cuda_lib):
    """Consecutive calls on one stream may overlap their launch and prologue
    (programmatic stream serialization): a call must read the previous
    call's output, and must not overwrite what the previous call still
    reads.  A chain of three calls, no synchronisation in between, on a
    shape small enough to leave most SMs idle:
      1. O1 = attn(Q, K, V)
      2. O2 = attn(O1, K, V)          reads O1 written by call 1
      3. attn(K2, K, V) written into Q's buffer, which call 1 read
    then O1 and O2 are checked against the oracle on the original inputs."""
    w = Workload("t", 1, 8, 512, 512, 64, "bf16", "BNSD", False, seed=31)
    x = make_inputs(w, device="cuda")
    q, k, v = x.q.clone(), x.k, x.v
    q_host = q.cpu()
    k2 = make_inputs(Workload("t2", 1, 8, 512, 512, 64, "bf16", "BNSD", False, seed=32),
                     device="cuda").q
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(1, 8, 512, device="cuda")
    l2, l3 = torch.empty_like(l1), torch.empty_like(l1)
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")

    def call(qq, oo, ll):
        if split:
            st = binding.fa_fwd_splitkv(qq.data_ptr(), k.data_ptr(), v.data_ptr(), oo.data_ptr(),
                                        ll.data_ptr(), 1, 8, 8, 512, 512, 64, w.softmax_scale,
                                        "BNSD", 0, "bf16", None, None, None, 2, ws.data_ptr(),
                                        ws.numel(), stream)
        else:
            st = binding.fa_fwd(qq.data_ptr(), k.data_ptr(), v.data_ptr(), oo.data_ptr(),
                                ll.data_ptr(), 1, 8, 512, 512, 64, w.softmax_scale, "BNSD", 0,
                                "bf16", None, None, None, stream)
        assert st == 0, binding.FA_STATUS.get(st)

    for _ in range(3):
        call(q, o1, l1)
        call(o1, o2, l2)
        call(k2, q, l3)
        torch.cuda.synchronize()
        assert binding.fa_last_device_error(stream) == 0
        O1, L1 = oracle.attention_full(q_host, x.k, x.v, dtype="bf16", layout="BNSD", B=1, H=8,
                                       S_q=512, S_kv=512, D=64, scale=w.softmax_scale,
                                       causal=False)
        assert float(np.abs(o1.float().cpu().double().numpy() - O1).max()) <= 1.6e-2
        assert float(np.abs(l1.cpu().double().numpy() - L1).max()) <= 1e-3
        O2, L2 = oracle.attention_full(o1.cpu(), x.k, x.v, dtype="bf16", layout="BNSD", B=1, H=8,
                                       S_q=512, S_kv=512, D=64, scale=w.softmax_scale,
                                       causal=False)
        assert float(np.abs(o2.float().cpu().double().numpy() - O2).max()) <= 1.6e-2
        assert float(np.abs(l2.cpu().double().numpy() - L2).max()) <= 1e-3
        q.copy_(q_host.to("cuda"))   # restore Q for the next round


@pytest.mark.gpu
def test_e4m3_and_bf16_calls_back_to_back(cuda_lib):
    """The e4m3 forward runs 512 threads (its O correction warpgroup), the
    16-bit one 384; chained on one stream with no synchronisation in between:
    a bf16 call reads the e4m3 call's O as its Q, then a second e4m3 call
    overwrites that O while the bf16 call may still be running.  Bit for bit
    against the same three calls synchronised one by one."""
    S, H, D = 512, 8, 128
    scale = 1.0 / math.sqrt(D)
    xa = make_inputs(Workload("t", 1, H, S, S, D, "e4m3", "BNSD", True, seed=33), device="cuda")
    xc = make_inputs(Workload("t", 1, H, S, S, D, "e4m3", "BNSD", False, seed=35), device="cuda")
    xb = make_inputs(Workload("t", 1, H, S, S, D, "bf16", "BNSD", False, seed=34), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    descale = lambda x: [torch.tensor([d], dtype=torch.float32, device="cuda") for d in x.descale]
    da, dc = descale(xa), descale(xc)

    def e4m3(x, d, o, lse, causal):
        st = binding.fa_fwd(x.q.data_ptr(), x.k.data_ptr(), x.v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), 1, H, S, S, D, scale, "BNSD", causal, "e4m3",
                            d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), stream)
        assert st == 0, binding.FA_STATUS.get(st)

    def bf16(q, o, lse):
        st = binding.fa_fwd(q.data_ptr(), xb.k.data_ptr(), xb.v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), 1, H, S, S, D, scale, "BNSD", 0, "bf16", None, None,
                            None, stream)
        assert st == 0, binding.FA_STATUS.get(st)

    def outputs():
        return (torch.empty(1, H, S, D, dtype=torch.bfloat16, device="cuda"),
                torch.empty(1, H, S, device="cuda"))

    (o1, l1), (o2, l2), (r1, rl1), (r2, rl2), (r3, rl3) = (outputs() for _ in range(5))
    e4m3(xa, da, r1, rl1, 1)
    torch.cuda.synchronize()
    bf16(r1, r2, rl2)
    torch.cuda.synchronize()
    e4m3(xc, dc, r3, rl3, 0)
    torch.cuda.synchronize()
    for _ in range(3):
        e4m3(xa, da, o1, l1, 1)
        bf16(o1, o2, l2)
        e4m3(xc, dc, o1, l1, 0)
        torch.cuda.synchronize()
        assert binding.fa_last_device_error(stream) == 0
        assert torch.equal(o2.view(torch.int16), r2.view(torch.int16)) and torch.equal(l2, rl2)
        assert torch.equal(o1.view(torch.int16), r3.view(torch.int16)) and torch.equal(l1, rl3)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_backward_calls_back_to_back(causal, cuda_lib):
    """The backward's dQ and dK/dV kernels are programmatic dependents of the
    launch before them (the dK/dV kernel may start while the dQ kernel still
    runs and waits for it only before it exits): work queued after a backward
    call must still see all of its outputs.  Two calls, no synchronisation in
    between: the second reads the first's dQ as its dO and writes its own dQ
    into the buffer the first read as dO.  Compared with the same two calls
    synchronised one by one; the backward is deterministic, so bit for bit."""
    B, H, S, D = 1, 8, 1024, 128
    w = Workload("t", B, H, S, S, D, "bf16", "BNSD", causal, seed=41)
    x = make_inputs(w, device="cuda")
    q, k, v = x.q, x.k, x.v
    stream = torch.cuda.current_stream().cuda_stream
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda")
    assert binding.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, S, S, D, w.softmax_scale, "BNSD", causal, "bf16", None, None,
                          None, stream) == 0
    st, nb = binding.fa_bwd_workspace_size(B, H, S)
    assert st == 0
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(42)
    do0 = (torch.randn(q.shape, generator=g, device="cuda") * 0.5).to(torch.bfloat16)

    def bwd(dout, dq, dk, dv):
        st = binding.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), B, H, H, S, S, D, w.softmax_scale, "BNSD", causal,
                            "bf16", ws.data_ptr(), nb, stream)
        assert st == 0, binding.FA_STATUS.get(st)

    def run(sync):
        do = do0.clone()
        dq1, dk1, dv1, dk2, dv2 = (torch.empty_like(q) for _ in range(5))
        torch.cuda.synchronize()
        bwd(do, dq1, dk1, dv1)
        if sync:
            torch.cuda.synchronize()
        bwd(dq1, do, dk2, dv2)          # dO = the first call's dQ; dQ into the first's dO
        torch.cuda.synchronize()
        assert binding.fa_last_device_error(stream) == 0
        return [t.clone() for t in (dq1, dk1, dv1, do, dk2, dv2)]

    ref = run(sync=True)
    for _ in range(3):
        got = run(sync=False)
        for name, a, b in zip(("dq1", "dk1", "dv1", "dq2", "dk2", "dv2"), got, ref):
            assert torch.equal(a, b), f"{name} differs from the synchronised calls"
        assert all(torch.isfinite(t.float()).all() for t in got)
