"""GB300 (sm_103a) Multiple-Item Scoring prefill hot path.

``ranking_prefill_gb300.lib`` binds the C-ABI shared library built from
``csrc/`` (``mis_attention_fwd``, ``mis_label_scores`` and the layout and
planning calls). Importing this package does not load the library; the
binding loads it on first use and raises if it is missing.
"""
__all__ = ["lib", "synth"]
