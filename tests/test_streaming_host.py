"""StreamingLayer's host logic on a stand-in context (no GPU): which library call each part of a
call goes to, what the C-token buffer holds when a chunk is committed, and when commits happen.
The stand-in records the calls and emulates the chunk-buffer stores of ipttt_decode_step."""
import pytest
import torch

from weight_mlp_layers_swiglu_b300.native import StreamingLayer

B, d, f, k, C = 2, 4, 6, 3, 8


class FakeCtx:
    def __init__(self):
        self.log = []

    def layer_forward(self, H, X0, W_gate, W_up, W_down0, W_target, conv_w, C_, eta):
        return torch.zeros(H.shape[0], 0, d), torch.zeros(H.shape[0], d, f)

    def layer_resume(self, H, X0, W_gate, W_up, W_target, conv_w, W_state, halo, C_, eta, O=None, W_state_out=None,
                     X0_halo_out=None):
        self.log.append(("resume", H.clone()))
        return torch.full((H.shape[0], H.shape[1], d), 1.0), W_state + 1.0, X0_halo_out

    def state_weight(self, state, dtype, W):
        self.log.append(("state_weight", float(state[0, 0, 0])))
        W.copy_(state.to(dtype))
        return W

    def swiglu(self, H2d, W_gate, W_up):
        self.log.append(("swiglu", H2d.shape[0]))
        return torch.zeros(H2d.shape[0], f)

    def chunk_apply(self, Z, W_eff, C_):
        self.log.append(("chunk_apply", Z.shape[1]))
        return torch.full((Z.shape[0], Z.shape[1], d), 2.0)

    def decode_step(self, H, W_gate, W_up, W_cur, X0=None, H_buf=None, X0_buf=None, pos=0):
        m = H.shape[1]
        self.log.append(("decode_step", m, pos))
        H_buf[:, pos:pos + m] = H
        X0_buf[:, pos:pos + m] = X0
        return torch.full((H.shape[0], m, d), 3.0), None


def _run(steps, exact=False, C=C):
    ctx = FakeCtx()
    W = torch.zeros(d, f)
    sl = StreamingLayer(ctx, torch.zeros(f, d), torch.zeros(f, d), W, torch.zeros(d, d), torch.zeros(d, k), B, C, 0.1,
                        exact=exact)
    T = sum(steps)
    H = torch.arange(B * T * d, dtype=torch.float32).reshape(B, T, d)
    outs, lo = [], 0
    for n in steps:
        outs.append(sl.step(H[:, lo:lo + n], H[:, lo:lo + n] * 10))
        lo += n
    sl.flush()
    return ctx.log, torch.cat(outs, dim=1), H, sl


def test_single_tokens_go_to_the_decode_step_and_commit_each_chunk():
    log, O, H, sl = _run([1] * 11)
    kinds = [e[0] for e in log]
    assert kinds == ["state_weight"] + ["decode_step"] * 8 + ["resume", "state_weight"] + ["decode_step"] * 3 + ["resume"]
    assert [e[2] for e in log if e[0] == "decode_step"] == list(range(8)) + [0, 1, 2]
    commits = [e[1] for e in log if e[0] == "resume"]
    assert torch.equal(commits[0], H[:, :8]) and torch.equal(commits[1], H[:, 8:11])
    assert torch.equal(O, torch.full((B, 11, d), 3.0))
    assert float(sl.state[0, 0, 0]) == 2.0  # two commits


def test_whole_chunks_resume_and_partials_fill_the_buffer():
    log, O, H, sl = _run([16, 3, 9, 4])
    kinds = [e[0] for e in log]
    # 16: two whole chunks; 3 and then 5 decode rows complete the third chunk, which is committed;
    # 4 and 4 more complete the fourth, committed at once (flush has nothing left)
    assert kinds == ["resume", "state_weight", "decode_step", "decode_step", "resume", "state_weight", "decode_step",
                     "decode_step", "resume"]
    assert [(e[1], e[2]) for e in log if e[0] == "decode_step"] == [(3, 0), (5, 3), (4, 0), (4, 4)]
    commits = [e[1] for e in log if e[0] == "resume"]
    assert torch.equal(commits[0], H[:, :16])
    assert torch.equal(commits[1], H[:, 16:24])
    assert torch.equal(commits[2], H[:, 24:32])
    assert O.shape == (B, 32, d)


def test_more_than_eight_partial_tokens_use_the_tensor_core_steps():
    log, O, H, sl = _run([3, 12], C=16)
    assert [e[0] for e in log] == ["state_weight", "decode_step", "swiglu", "chunk_apply", "resume"]
    assert torch.equal([e[1] for e in log if e[0] == "resume"][0], H[:, :15])  # flush commits the partial chunk
    assert torch.equal(O[:, 3:], torch.full((B, 12, d), 2.0))


def test_exact_mode_keeps_the_tensor_core_steps():
    log, O, H, sl = _run([1] * 3, exact=True)
    assert [e[0] for e in log] == ["state_weight"] + ["swiglu", "chunk_apply"] * 3 + ["resume"]
    assert torch.equal([e[1] for e in log if e[0] == "resume"][0], H[:, :3])
