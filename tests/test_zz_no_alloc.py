"""The attention entry point that allocates nothing (tfl_attention_decode_noalloc),
for callers that cannot allocate device memory where they run attention.  It must
give what the workspace-backed attention (tfl_layer_op "attention") gives, call
after call, although every call reuses the same fixed scratch array."""
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    tfl.lib()


def _attention_only_model(shape, max_context):
    """A model whose weights are small stand-ins: attention reads only q and the cache."""
    z = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    w = {k: z for k in ("embed", "final_norm")}
    w["lm_head"] = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    for k in synth.LAYER_KEYS:
        w[k] = [torch.zeros(64, dtype=torch.bfloat16, device="cuda") for _ in range(shape.layers)]
    return tfl.Model(shape, w, max_rows=16, max_decode_rows=16, max_context=max_context)


@pytest.mark.parametrize("shape", [synth.TINY.with_layers(2), synth.NANBEIGE_33B.with_layers(2)],
                         ids=["tiny", "33b"])
def test_noalloc_attention_matches_workspace_attention_twice(shape):
    ctx = 1000
    m = _attention_only_model(shape, ctx + 64)
    kv = m.kv(ctx + 64)
    for l in range(shape.layers):
        K, V = synth.kv_contents(shape, 70, l, ctx + 16, "cuda")
        kv.write(l, 0, K, V)
    qd = shape.n_q * shape.head_dim
    # two calls in a row with different rows, positions and layers: the shared
    # scratch of the first call must not leak into the second
    for call, (layer, pos0, R) in enumerate([(1, ctx, 5), (0, ctx - 300, 16)]):
        q = synth.normal_bf16(71 + call, 0, (R, qd), 1.5, "cuda")
        ref = torch.empty((R, qd), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_layer_op(m, "attention", layer, q, ref, kv, pos0)
        out = torch.full((R, qd), float("nan"), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_attention_decode_noalloc(kv, layer, pos0, q, out)
        torch.cuda.synchronize()
        gu.assert_hidden_gate(synth.bits(out), synth.bits(ref), f"call {call}")
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "same kernels, same inputs"


def test_noalloc_attention_refuses_sizes_beyond_its_scratch():
    shape = synth.NANBEIGE_33B.with_layers(1)
    m = _attention_only_model(shape, 20480)
    kv = m.kv(20480)
    q = torch.zeros((16, shape.n_q * 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(tfl.TflError) as e:
        tfl.tfl_attention_decode_noalloc(kv, 0, 20000, q, out)   # 16 rows x 56 heads x 40 units of 512 keys
    assert e.value.code == tfl.TFL_E_WORKSPACE and "16 MiB" in str(e.value)


def test_noalloc_attention_near_its_limit():
    """One 33B-shaped row at position 294,900: 56 heads x 576 units of 512 keys =
    32,256 partials of the 32,263 the scratch holds; bit-equal to the workspace
    attention on the same inputs."""
    shape = synth.NANBEIGE_33B.with_layers(1)
    pos0 = 294900
    m = _attention_only_model(shape, pos0 + 64)
    kv = m.kv(pos0 + 64)
    K, V = synth.kv_contents(shape, 72, 0, pos0 + 1, "cuda")
    kv.write(0, 0, K, V)
    del K, V
    qd = shape.n_q * shape.head_dim
    q = synth.normal_bf16(73, 0, (1, qd), 1.7, "cuda")
    ref = torch.empty((1, qd), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_layer_op(m, "attention", 0, q, ref, kv, pos0)
    out = torch.full((1, qd), float("nan"), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_attention_decode_noalloc(kv, 0, pos0, q, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
