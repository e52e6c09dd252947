"""Host-side logic of bench.py (no GPU): the launch count it claims per
step, and the comment-insensitive source hash that ties an ncu traffic
record to the code it was measured on."""
from types import SimpleNamespace

import bench

LM, FACT = 0x1, 0x2


class FakeState:
    def __init__(self, recipe, slots):
        self.recipe = recipe
        self.slots = [SimpleNamespace(numel=n, rows=r, flags=f) for n, r, f in slots]

    def is_factored(self, sl):
        return self.recipe == "factored" and bool(sl.flags & FACT) and sl.numel > 0 and sl.numel % sl.rows == 0


def test_launches_per_step():
    plain = FakeState("zip_sr", [(4096, 1, 0), (1024 * 64, 64, 0), (256 * 8, 256, LM)])
    assert bench.launches_per_step(plain) == 1
    assert bench.launches_per_step(plain, flags=0x1) == 2             # LM head on its own launch
    assert bench.launches_per_step(plain, flags=0x2) == 1             # every tensor rounds m stochastically
    assert bench.launches_per_step(plain, clip=True) == 4             # + sum of squares (3 kernels)
    tao = FakeState("torchao", [(4096, 1, 0), (256 * 8, 256, LM)])
    assert bench.launches_per_step(tao, flags=0x1) == 1               # TorchAO keeps RTN on the head
    fac = FakeState("factored", [(1024 * 64, 64, FACT), (1024, 1, 0)])
    assert bench.launches_per_step(fac) == 1 + 1 + 4                  # two step launches + statistics
    fac_only = FakeState("factored", [(1024 * 64, 64, FACT)])
    assert bench.launches_per_step(fac_only) == 1 + 4


def test_strip_comments_keeps_code_and_literals():
    src = 'int a = 1; // trailing\n/* block\n comment */ const char* s = "// kept /* too */";\n  char q = \'"\';  int   b;'
    out = bench._strip_comments(src)
    assert out == 'int a = 1; const char* s = "// kept /* too */"; char q = \'"\'; int b;'
    assert bench._strip_comments("a /* x */ b // y\nc") == bench._strip_comments("a b\n   c")
    assert bench._strip_comments("a+b") != bench._strip_comments("a-b")


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()


def test_companion_workload_only_beside_the_plain_default():
    def args(**kw):
        base = dict(companion="auto", workload="llama8b_zipsr", tensors=0, tensor_slice="", variant="none",
                    max_grad_norm=None)
        base.update(kw)
        return SimpleNamespace(**base)
    assert bench.companion_workload(args()) == "llama8b_zeeden"
    assert bench.companion_workload(args(companion="none")) is None
    assert bench.companion_workload(args(workload="llama8b_zeeden")) is None
    assert bench.companion_workload(args(tensor_slice="1:10")) is None
    assert bench.companion_workload(args(variant="m_sr_all")) is None
    assert bench.companion_workload(args(max_grad_norm=1.0)) is None
    assert bench.companion_workload(args(companion="gpt1p4b_zipsr", workload="qwen0p6b_factored")) == "gpt1p4b_zipsr"
