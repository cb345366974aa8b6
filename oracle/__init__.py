"""Plain, slow CPU oracle for the TurboQuant hot path (fp64 NumPy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA/C++ path; the two
sides meet only through the seeded synthetic inputs of
``decode_attention_21_b300.workloads`` and through the documented byte layout
of the packed cache.

Sources (web pages describing Google Research's TurboQuant, arXiv 2504.19874):

* [xujun] xujun.org note-189244, "TurboQuant ... 两步绝杀" — sections
  "第一步：PolarQuant", "第二步：QJL", "性能数据".
* [suzuke] suzuke.github.io "TurboQuant: compressing AI consciousness" —
  section "技術上怎麼做到的" (第一步 / 第二步 / 第三步) and "實際跑出來的數據".
* [cnyes] hao.cnyes.com "TurboQuant" (AGI-Hunt explainer) — "極坐標的妙用",
  "1 bit 掃尾", "高精度的那一側「兜住了」".

Modules:
    rng        counter-based splitmix64 + Box-Muller (shared generator definition)
    codebook   Lloyd-Max solver on the rotated-coordinate density
    rotation   seeded Haar rotation Pi (QR of a Gaussian matrix)
    quant      scalar stage 1, QJL residual sketch, mixed-bit variant
    polar      recursive-polar stage 1
    layout     packed bit-plane cache byte layout (pack / unpack)
    estimate   inner-product estimator, logits, decode attention, top-k search
    split      outlier-channel split: independent instances per channel group
"""
from . import rng, codebook, rotation, quant, polar, layout, estimate, split  # noqa: F401
