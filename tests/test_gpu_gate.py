"""GPU tests of dsv4_stream_gate (pipelined input staging): flags set by a
copy stream open the gate and are cleared; a flag nothing sets runs the
bounded wait out and reports it; a staged loop (inputs copied on one stream,
the gate and a kernel that reads them on another, results read back on a
third) computes every step from that step's own inputs."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import dev

pytestmark = pytest.mark.gpu


def test_gate_opens_on_set_flags_and_clears_them():
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    one = torch.ones(1, dtype=torch.int32).pin_memory()
    s_in = torch.cuda.Stream()
    with torch.cuda.stream(s_in):
        flags[0:1].copy_(one, non_blocking=True)
        flags[2:3].copy_(one, non_blocking=True)
    B.stream_gate([flags[0:1], flags[2:3]], status=status)
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    assert flags.cpu().tolist() == [0, 0, 0, 0]


def test_gate_wait_runs_out_and_reports_it():
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags[1] = 1
    B.stream_gate([flags[0:1], flags[1:2]], status=status, timeout_us=100000)     # flag 0: nothing sets it
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.ERR_TIMEOUT and bits & B.DEV_TIMEOUT
    assert flags.cpu().tolist() == [0, 1]                 # a wait that ran out clears nothing
    # the context stays usable: the gate opens on the flag once it is set
    flags[0] = 1
    B.stream_gate([flags[0:1]], status=status)
    torch.cuda.synchronize()
    assert B.read_device_status(status)[0] == B.OK
    assert flags.cpu().tolist() == [0, 1]


@pytest.mark.parametrize("graph", [False, True])
def test_staged_loop_reads_each_steps_own_inputs(graph):
    """Steps alternate between two device input blocks and two output blocks.
    Inputs (bf16 attention outputs and positions) are copied on one stream,
    which then sets the block's input flag; the compute stream runs the gate
    on (input flag, output-read flag) and the output quantisation; a third
    stream reads the codes back and sets the output-read flag.  No compute-
    stream event waits.  Every step's codes equal the oracle's quantisation
    of that step's inputs."""
    T, H, steps = 4, 16, 12
    g = synth.rng(81)
    cs = oracle.rope_table(4096, 64)
    cs_d = dev(cs)
    o_bits = [oracle.f32_to_bf16(synth.normal(g, (T * H, 512), 0.1)).reshape(T, H, 512) for _ in range(steps)]
    pos = [g.integers(0, 4096, size=T).astype(np.int32) for _ in range(steps)]
    host_o = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in o_bits]
    host_p = [torch.from_numpy(p).pin_memory() for p in pos]
    host_codes = [torch.empty((T, H, 512), dtype=torch.uint8).pin_memory() for _ in range(steps)]
    d_o = [torch.empty((T, H, 512), dtype=torch.int16, device="cuda") for _ in range(2)]
    d_p = [torch.empty(T, dtype=torch.int32, device="cuda") for _ in range(2)]
    d_codes = [torch.empty((T, H, 512), dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_scales = [torch.empty((T, H, 4), dtype=torch.float32, device="cuda") for _ in range(2)]
    host_scales = [torch.empty((T, H, 4), dtype=torch.float32).pin_memory() for _ in range(steps)]
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")      # in[0], in[1], out_read[0], out_read[1]
    flags[2:] = 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    one = torch.ones(1, dtype=torch.int32).pin_memory()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()

    def loop():
        s_c = torch.cuda.current_stream()
        s_in.wait_stream(s_c)
        s_out.wait_stream(s_c)
        done = [None, None]
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if done[b] is not None:
                    s_in.wait_event(done[b])
                d_o[b].copy_(host_o[i], non_blocking=True)
                d_p[b].copy_(host_p[i], non_blocking=True)
                flags[b:b + 1].copy_(one, non_blocking=True)
            B.stream_gate([flags[b:b + 1], flags[2 + b:3 + b]], status=status)
            B.inv_rope_fp8_quant(d_o[b].view(torch.bfloat16), d_p[b], cs_d, d_codes[b], d_scales[b], status=status)
            ev = torch.cuda.Event()
            ev.record(s_c)
            done[b] = ev
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                host_codes[i].copy_(d_codes[b], non_blocking=True)
                host_scales[i].copy_(d_scales[b], non_blocking=True)
                flags[2 + b:3 + b].copy_(one, non_blocking=True)
        s_c.wait_stream(s_in)
        s_c.wait_stream(s_out)

    if graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            loop()
        for c in host_codes:
            c.fill_(0xAA)
        gr.replay()
    else:
        loop()
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    for i in range(steps):
        for t in range(T):
            wc, ws = oracle.inv_rope_fp8_quant(o_bits[i][t], int(pos[i][t]), cs)
            assert np.array_equal(host_codes[i].numpy()[t], wc), "step %d token %d" % (i, t)
            assert np.array_equal(host_scales[i].numpy()[t].view(np.uint32), ws.view(np.uint32))
    assert flags.cpu().tolist() == [0, 0, 1, 1]
