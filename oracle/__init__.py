"""CPU oracle for MoE expert routing with equal-cost load balancing.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import, call or run anything in
this package; the library (``moe_expert_routing_router_gb300``) never does, and it
shares no code, table or helper with it.  Inputs come from ``synth`` (seeded
generators that hold none of the method's arithmetic).

Everything is plain numpy in float64, single-threaded, written to be read
against the source pages:

  [P1] the three-layer load-balancing article (LVS, NIC Teaming, MoE
       equal-cost balancing), mhpq.cn/news/998159
  [P2] "MoE大模型训练中的等开销负载均衡：原理、代码实现与调参实战", codechina.net
  [P3] the large-model load-balancing survey printed under the title
       "企业官网建设流程全解析", cnvsn.com/news/335486
  [P4] "MoE 训练端到端加速 1.43 倍：LoongForge 基于拓扑感知最优传输重新定义 EP
       专家负载均衡", LoongForge blog (TAOT)

Modules:
  router    -- softmax, top-k, gates, f_i, P_i, L_aux, CV, per-rank loads, dL_aux/dlogits
  dispatch  -- capacity and the stable capacity-limited token->expert dispatch
  sinkhorn  -- TAOT Phase 1: topology-aware entropic transport plan
  routing_ext -- aux-loss-free bias routing, masked P_i, the full backward through the gates
  eplb      -- EPLB expert replication and balanced packing onto GPUs ([P3] §4.1.2)
  taot_match -- TAOT Phase 2: column-first matching of hot experts to cold ranks ([P4] §2)

Parity status of each function is stated in its docstring ("pinned by ...");
the pins live in ``tests/test_oracle_*.py``.
"""

from . import router, dispatch, sinkhorn, routing_ext, eplb, taot_match  # noqa: F401
