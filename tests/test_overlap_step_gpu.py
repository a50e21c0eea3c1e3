"""A data-parallel training step on one GPU through the pieces a trainer
uses: backward with GradReduceOverlap's hooks (world 1: the buffers only),
then MuonWithAdamW on the reduced gradients (matrices through muon_step,
the rest through muon_adamw_step).  The parameters must equal, bit for bit,
those of a plain backward followed by the same optimizer step."""
import pytest
import torch

from helpers import muon

pytestmark = pytest.mark.gpu


class _Net(torch.nn.Module):
    """Two linear layers and a layer norm; the output projection reuses the
    first layer's weight (a tied weight).  Every op has a deterministic
    backward, so two equal nets get equal gradients."""

    def __init__(self):
        super().__init__()
        g = torch.Generator().manual_seed(3)
        self.l1 = torch.nn.Linear(128, 256)
        self.ln = torch.nn.LayerNorm(256)
        self.l2 = torch.nn.Linear(256, 128)
        with torch.no_grad():
            for p in self.parameters():
                p.copy_(torch.randn(p.shape, generator=g) * 0.05)

    def forward(self, x):
        h = self.ln(torch.relu(self.l1(x)))
        return self.l2(h) @ self.l1.weight.t()


def _loss(net, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(128, 128, generator=g, device="cuda").to(torch.bfloat16)
    y = torch.randint(0, 256, (128,), generator=g, device="cuda")
    return torch.nn.functional.cross_entropy(net(x).float(), y)


def test_overlapped_reduction_then_muon_with_adamw_step():
    m = muon()
    from newton_schulz_05_gb300.comm import GradReduceOverlap
    nets = [_Net().cuda().to(torch.bfloat16) for _ in range(2)]
    opts = [m.MuonWithAdamW(list(n.parameters()), lr=0.02, adamw_lr=1e-3) for n in nets]
    ov = GradReduceOverlap(list(nets[0].parameters()), bucket_bytes=64 << 10)
    for step in range(3):
        ov.begin()
        _loss(nets[0], step).backward()
        grads = ov.finish()
        opts[0].step(grads)
        _loss(nets[1], step).backward()
        opts[1].step([p.grad for p in nets[1].parameters()])
        for p in nets[1].parameters():
            p.grad = None
        torch.cuda.synchronize()
        for a, b in zip(nets[0].parameters(), nets[1].parameters()):
            assert torch.equal(a, b), "step %d" % step
    assert len(ov.buckets) >= 3
