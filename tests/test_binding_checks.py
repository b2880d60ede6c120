"""The Python binding's argument checks (no GPU): element types, shapes and
layouts the C ABI cannot see behind a raw pointer are rejected before
anything reaches the library, and correctly typed and shaped tensors pass
every check up to the last one, that the memory is on the device."""
import pytest
import torch

from mla_tree_verify_ddt_gb300 import ddtree

B, D, K, BUDGET, H, TCAP, V = 2, 3, 4, 8, 4, 40, 64
QC = BUDGET + 1


def t(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


def tree():
    return ddtree.Tree.empty(B, D, BUDGET, "cpu")


def attn_args():
    return [t(B, QC, H, 512, dtype=torch.bfloat16), t(B, QC, H, 64, dtype=torch.bfloat16),
            t(B, TCAP, 512, dtype=torch.bfloat16), t(B, TCAP, 64, dtype=torch.bfloat16),
            t(B, dtype=torch.int32)]


def accept():
    i32 = torch.int32
    return ddtree.Accept(t(B, dtype=i32), t(B, D + 1, dtype=i32), t(B, D + 1, dtype=i32), t(B, dtype=i32))


def only_device_missing(fn):
    with pytest.raises(ValueError, match="CUDA tensors"):
        fn()


def test_valid_arguments_pass_every_check_but_the_device():
    i32 = torch.int32
    only_device_missing(lambda: ddtree.ddt_tree_build(t(B, D, K, dtype=i32), t(B, D, K), t(B, dtype=i32),
                                                      BUDGET, V))
    only_device_missing(lambda: ddtree.ddt_verify_mla_attn(*attn_args(), tree(), 0.07))
    only_device_missing(lambda: ddtree.ddt_verify_mla_attn_bf16(*attn_args(), tree(), 0.07))
    only_device_missing(lambda: ddtree.ddt_verify_mla_attn_noalloc(*attn_args(), tree(), 0.07))
    a = attn_args()
    only_device_missing(lambda: ddtree.ddt_verify_mla_attn_paged(
        a[0], a[1], t(100, 512, dtype=torch.bfloat16), t(100, 64, dtype=torch.bfloat16), a[4],
        t(B, TCAP, dtype=i32), tree(), 0.07))
    only_device_missing(lambda: ddtree.ddt_tree_accept(tree(), t(B, QC, dtype=i32)))
    only_device_missing(lambda: ddtree.ddt_kv_commit(accept(), t(B, TCAP, 512, dtype=torch.int16),
                                                     t(B, TCAP, 64, dtype=torch.int16), t(B, dtype=i32),
                                                     t(B, dtype=i32)))
    only_device_missing(lambda: ddtree.ddt_tree_sample(tree(), t(B, QC, V), 1.0, t(B, QC)))
    only_device_missing(lambda: ddtree.VerifyStep(t(B, D, K, dtype=i32), t(B, D, K), t(B, dtype=i32), V,
                                                  BUDGET, *attn_args(), t(B, QC, dtype=i32), 0.07,
                                                  acc=accept()))


@pytest.mark.parametrize("which,bad", [
    (0, t(B, QC, H, 512, dtype=torch.float16)),    # q_lat not bfloat16
    (2, t(B, TCAP, 512)),                          # c_kv float32
    (4, t(B, dtype=torch.int64)),                  # prefix_len int64
])
def test_attention_rejects_wrong_element_types(which, bad):
    a = attn_args()
    a[which] = bad
    with pytest.raises(TypeError):
        ddtree.ddt_verify_mla_attn(*a, tree(), 0.07)


@pytest.mark.parametrize("which,bad", [
    (0, t(B, QC, H, 576, dtype=torch.bfloat16)),   # latent width
    (1, t(B, QC, H + 1, 64, dtype=torch.bfloat16)),  # heads differ from q_lat's
    (2, t(B + 1, TCAP, 512, dtype=torch.bfloat16)),  # batch differs from the tree's
    (3, t(B, TCAP - 1, 64, dtype=torch.bfloat16)),   # key capacity differs from c_kv's
])
def test_attention_rejects_wrong_shapes(which, bad):
    a = attn_args()
    a[which] = bad
    with pytest.raises(ValueError, match="shape"):
        ddtree.ddt_verify_mla_attn(*a, tree(), 0.07)


def test_non_dense_tensors_are_rejected():
    a = attn_args()
    a[2] = t(B, 512, TCAP, dtype=torch.bfloat16).transpose(1, 2)
    with pytest.raises(ValueError, match="dense"):
        ddtree.ddt_verify_mla_attn(*a, tree(), 0.07)


def test_outputs_and_accept_buffers_are_checked():
    with pytest.raises(TypeError):
        ddtree.ddt_verify_mla_attn(*attn_args(), tree(), 0.07, out=t(B, QC, H, 512, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        ddtree.ddt_verify_mla_attn_bf16(*attn_args(), tree(), 0.07, out=t(B, QC, H, 512))
    bad = accept()
    bad.accept_idx = t(B, D, dtype=torch.int32)    # D entries instead of D + 1
    with pytest.raises(ValueError, match="shape"):
        ddtree.ddt_tree_accept(tree(), t(B, QC, dtype=torch.int32), out=bad)
    with pytest.raises(TypeError):
        ddtree.ddt_tree_sample(tree(), t(B, QC, V, dtype=torch.float64), 1.0)
    with pytest.raises(TypeError):
        ddtree.ddt_kv_commit(accept(), t(B, TCAP, 512), t(B, TCAP, 64), t(B, dtype=torch.int32),
                             t(B, dtype=torch.int32))


class _FakeCuda:
    """Stands in for a CUDA tensor or stream on device `index` (only the
    attributes the device check reads)."""

    def __init__(self, index):
        self.is_cuda = True
        self.device = torch.device("cuda", index)


def test_tensors_of_another_device_are_rejected(monkeypatch):
    # the library launches on the current device: cuda:0 here
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    ddtree._on_device(_FakeCuda(0), None, _FakeCuda(0), stream=_FakeCuda(0))
    with pytest.raises(ValueError, match="current CUDA device"):
        ddtree._on_device(_FakeCuda(0), _FakeCuda(1))
    with pytest.raises(ValueError, match="current CUDA device"):
        ddtree._on_device(_FakeCuda(1))
    with pytest.raises(ValueError, match="stream of cuda:1"):
        ddtree._on_device(_FakeCuda(0), stream=_FakeCuda(1))
    with pytest.raises(ValueError, match="CUDA tensors"):
        ddtree._on_device(_FakeCuda(0), t(3))
