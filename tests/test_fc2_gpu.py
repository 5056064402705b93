"""GPU parity of the FlashComm2 token reorganisation (sp_fc2_reorganize) with the oracle's
step-by-step simulation (vllm-ascend SP/FlashComm notes §4.4): bit-exact, every output byte
written, no byte written outside y."""
import numpy as np
import pytest
import torch

import oracle
import sequence_reduce_add_gb300 as sp

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096


@pytest.mark.parametrize("G,P,N,H,dtype", [
    (4, 2, 4 * 16, 4 * 64, torch.bfloat16),        # the page's tp=4 / otp=2 shape, small
    (8, 2, 8 * 64, 8 * 896, torch.bfloat16),       # H = 7168
    (8, 4, 8 * 33, 8 * 512, torch.bfloat16),       # odd tokens per segment
    (16, 4, 16 * 7, 16 * 64, torch.bfloat16),
    (8, 8, 8 * 10, 8 * 128, torch.bfloat16),       # otp = global tp: identity
    (4, 1, 4 * 9, 4 * 256, torch.bfloat16),        # otp = 1: each rank gets whole rows
    (8, 2, 8 * 40, 8 * 64, torch.uint8),           # 1-byte elements (e.g. FP8 activations)
    (8, 2, 8 * 40, 8 * 32, torch.float32),
    (8, 2, 8 * 512, 8 * 896, torch.bfloat16),      # 4096 tokens, H = 7168
    (8, 2, 8 * 1400, 8 * 256, torch.bfloat16),     # several ring passes per CTA
    (4, 2, 4 * 3, 4 * 8, torch.bfloat16),          # 16-byte pieces, one ragged tile
    (2, 1, 2 * 5, 2 * 8704, torch.bfloat16),       # pieces larger than a ring stage
])
def test_fc2_reorganize_matches_oracle(G, P, N, H, dtype):
    D = G // P
    F = H // G
    g = torch.Generator(device=DEV).manual_seed(G * 1000 + P * 100 + N)
    x = torch.randint(0, 255, (G, N, F * torch.empty((), dtype=dtype).element_size()),
                      generator=g, device=DEV, dtype=torch.uint8).view(dtype)
    ybytes = G * (N // D) * D * F * x.element_size()
    outs = []
    for fill in (0xA5, 0x5A):
        whole = torch.full((ybytes + 2 * GUARD,), 0xC3, dtype=torch.uint8, device=DEV)
        whole[GUARD:GUARD + ybytes].fill_(fill)
        y = whole[GUARD:GUARD + ybytes].view(dtype).view(G, N // D, D * F)
        sp.sp_fc2_reorganize(x, P, y)
        torch.cuda.synchronize()
        guard = torch.cat([whole[:GUARD], whole[-GUARD:]])
        assert bool((guard == 0xC3).all()), "write outside y"
        outs.append(y.cpu())
    assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8)), "unwritten bytes"
    ref = oracle.fc2_reorganize(x.cpu().view(torch.uint8).numpy().reshape(G, N, -1)
                                .view(np.dtype(f"u{x.element_size()}")) if x.element_size() in (1, 2, 4)
                                else x.cpu().numpy(), P)
    got = outs[0].view(torch.uint8).numpy().reshape(ref.shape[0], ref.shape[1], -1)
    assert np.array_equal(got, ref.view(np.uint8).reshape(got.shape))


def test_fc2_reads_what_the_fused_stage_just_wrote():
    """Fused stage then reorganisation on one stream, both launched with programmatic dependent
    launch: the reorganisation reads the new residual the fused call has just written (it must
    wait for that grid), in a loop and replayed from a CUDA graph."""
    from sequence_reduce_add_gb300 import synth
    w = synth.workload(2)
    inp = synth.make_inputs(w, device=DEV, T_pad=1024, T_valid=1024)
    G, P, F = 8, 2, 512
    N = 1024 * 4096 // (G * F)
    D = G // P
    res_out = torch.empty((1024, 4096), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(res_out)
    y = torch.empty((G, N // D, D * F), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()  # the inputs are written on torch's stream; `s` does not wait for it

    def step():
        sp.sp_fused_reduce_norm(inp["partials"], inp["weight"], out, res_out,
                                residual=inp["residual"], bias=inp["bias"], stream=s)
        sp.sp_fc2_reorganize(res_out.view(G, N, F), P, y, stream=s)

    def check():
        torch.cuda.synchronize()
        x = res_out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(G, N, F)
        ref = oracle.fc2_reorganize(x, P)
        assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), ref)

    for k in range(5):
        inp["partials"].mul_(0.5 if k % 2 else 2.0)   # new contents every step
        torch.cuda.current_stream().synchronize()
        step()
        check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        step()
    inp["residual"].mul_(-1.0)
    torch.cuda.synchronize()
    g.replay()
    check()
