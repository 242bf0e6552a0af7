"""Parameter shape lists of the synthetic workloads.

Each function returns the model's parameters in *registration order*
(the order ``module.parameters()`` would yield them), as a list of
``(name, shape)`` pairs.  Only shapes are produced: no weights, no data.

The models are the ones the DDP pages evaluate or print:

* ``linear_10x10`` -- the ``nn.Linear(10, 10)`` of the worked example on
  "Distributed Data Parallel" (tensorplay.cn notes, section "Example").
* ``resnet50`` / ``bert_large`` -- the two models of "PyTorch Distributed:
  Experiences on Accelerating Data Parallel Training" (evaluation, Section
  5), rebuilt from their published hyperparameters.
* ``gpt2_medium`` -- a 24-layer, d=1024, vocab-50257 decoder used for the
  bf16 bucket-cap sweep.
* ``uniform`` -- the equal-size tensor lists of the bucket-layout table on
  "NCCL 专家课程 30: DDP Reducer、Bucket 与计算通信重叠" (section
  "参数粒度实验"): 48 x 1 MiB and 12 x 4 MiB fp32 tensors.

This module holds no reducer arithmetic; it is shared input definition.
"""

from __future__ import annotations

from math import prod

Shape = tuple


def linear_10x10():
    """nn.Linear(10, 10): weight registered before bias."""
    return [("weight", (10, 10)), ("bias", (10,))]


def resnet50(num_classes: int = 1000):
    """ResNet-50 (bottleneck 3/4/6/3, expansion 4) with BatchNorm affine params.

    Registration order inside a bottleneck: conv1, bn1, conv2, bn2, conv3,
    bn3, then the downsample conv + bn of the first block of each stage.
    """
    out = [("conv1.weight", (64, 3, 7, 7)), ("bn1.weight", (64,)), ("bn1.bias", (64,))]
    inplanes = 64
    for stage, (planes, blocks) in enumerate([(64, 3), (128, 4), (256, 6), (512, 3)], start=1):
        for i in range(blocks):
            p = f"layer{stage}.{i}."
            out += [
                (p + "conv1.weight", (planes, inplanes, 1, 1)),
                (p + "bn1.weight", (planes,)), (p + "bn1.bias", (planes,)),
                (p + "conv2.weight", (planes, planes, 3, 3)),
                (p + "bn2.weight", (planes,)), (p + "bn2.bias", (planes,)),
                (p + "conv3.weight", (planes * 4, planes, 1, 1)),
                (p + "bn3.weight", (planes * 4,)), (p + "bn3.bias", (planes * 4,)),
            ]
            if i == 0:
                out += [
                    (p + "downsample.0.weight", (planes * 4, inplanes, 1, 1)),
                    (p + "downsample.1.weight", (planes * 4,)),
                    (p + "downsample.1.bias", (planes * 4,)),
                ]
            inplanes = planes * 4
    out += [("fc.weight", (num_classes, 2048)), ("fc.bias", (num_classes,))]
    return out


def bert_large(layers: int = 24, hidden: int = 1024, ffn: int = 4096,
               vocab: int = 30522, max_pos: int = 512, type_vocab: int = 2):
    """BERT-large encoder + pooler (no MLM head)."""
    h, f = hidden, ffn
    out = [
        ("embeddings.word_embeddings.weight", (vocab, h)),
        ("embeddings.position_embeddings.weight", (max_pos, h)),
        ("embeddings.token_type_embeddings.weight", (type_vocab, h)),
        ("embeddings.LayerNorm.weight", (h,)), ("embeddings.LayerNorm.bias", (h,)),
    ]
    for i in range(layers):
        p = f"encoder.layer.{i}."
        for m in ("query", "key", "value"):
            out += [(p + f"attention.self.{m}.weight", (h, h)), (p + f"attention.self.{m}.bias", (h,))]
        out += [
            (p + "attention.output.dense.weight", (h, h)), (p + "attention.output.dense.bias", (h,)),
            (p + "attention.output.LayerNorm.weight", (h,)), (p + "attention.output.LayerNorm.bias", (h,)),
            (p + "intermediate.dense.weight", (f, h)), (p + "intermediate.dense.bias", (f,)),
            (p + "output.dense.weight", (h, f)), (p + "output.dense.bias", (h,)),
            (p + "output.LayerNorm.weight", (h,)), (p + "output.LayerNorm.bias", (h,)),
        ]
    out += [("pooler.dense.weight", (h, h)), ("pooler.dense.bias", (h,))]
    return out


def gpt2_medium(layers: int = 24, d: int = 1024, vocab: int = 50257, n_ctx: int = 1024):
    """GPT-2 medium decoder (Conv1D weights stored in x out)."""
    out = [("wte.weight", (vocab, d)), ("wpe.weight", (n_ctx, d))]
    for i in range(layers):
        p = f"h.{i}."
        out += [
            (p + "ln_1.weight", (d,)), (p + "ln_1.bias", (d,)),
            (p + "attn.c_attn.weight", (d, 3 * d)), (p + "attn.c_attn.bias", (3 * d,)),
            (p + "attn.c_proj.weight", (d, d)), (p + "attn.c_proj.bias", (d,)),
            (p + "ln_2.weight", (d,)), (p + "ln_2.bias", (d,)),
            (p + "mlp.c_fc.weight", (d, 4 * d)), (p + "mlp.c_fc.bias", (4 * d,)),
            (p + "mlp.c_proj.weight", (4 * d, d)), (p + "mlp.c_proj.bias", (d,)),
        ]
    out += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return out


def uniform(count: int, numel: int):
    """``count`` independent tensors of ``numel`` elements each."""
    return [(f"p{i}", (numel,)) for i in range(count)]


def numels(shapes) -> list[int]:
    """Element count of each tensor of a shape list."""
    return [int(prod(s)) for _, s in shapes]


MIB = 1 << 20

# Named workloads: (shape-list factory, W, grad dtype, cap in MiB, ready order kind)
WORKLOADS = {
    "linear": dict(shapes=linear_10x10, W=2, dtype="f32", caps_mib=[25], order="reverse"),
    "resnet50": dict(shapes=resnet50, W=8, dtype="f32", caps_mib=[25], order="reverse"),
    "bert_large": dict(shapes=bert_large, W=4, dtype="f32", caps_mib=[25], order="straggler"),
    "gpt2_medium": dict(shapes=gpt2_medium, W=8, dtype="bf16", caps_mib=[0, 1, 5, 25, 100], order="reverse"),
    "nosync_resnet50": dict(shapes=resnet50, W=16, dtype="f32", caps_mib=[25], order="reverse", K=8),
}
